// The host-buffer pipeline shared by the *_host entry points: chunks of
// independent rows or samples are copied in on an internal stream, computed
// on the caller's stream and copied out on a second internal stream, through
// two device staging buffers each way, so that the copies of one chunk
// overlap the compute of its neighbours.
#pragma once

#include <cuda_runtime.h>

#include "host_common.h"

namespace gf {

// The pipeline's schedule, kept apart from the CUDA calls that carry it out,
// so that its error path can be run without a GPU.  Chunk i uses staging
// buffer i % 2: its copy-in waits until the compute of chunk i - 2 has read
// that buffer, its compute waits for its own copy-in and for the copy-out of
// chunk i - 2 (same output buffer), its copy-out waits for its compute.
// Every step returns false when one of its CUDA calls fails; then nothing
// more is enqueued and drain() blocks until the copies already queued on the
// internal streams have finished, so that none of them touches the caller's
// host buffers after the call returns.
struct HostPipeOps {
  virtual bool setup() = 0;                  // work every chunk needs, on the caller's stream
  virtual bool copy_in(int64_t i, int buf) = 0;
  virtual bool compute(int64_t i, int buf) = 0;
  virtual bool copy_out(int64_t i, int buf) = 0;
  virtual bool join() = 0;                   // the caller's stream waits for the last copy-outs
  virtual void drain() = 0;                  // error path: wait for everything already queued
  virtual ~HostPipeOps() = default;
};

inline gf_status run_host_pipeline(HostPipeOps& ops, int64_t nchunks) {
  bool ok = ops.setup();
  for (int64_t i = 0; ok && i < nchunks; ++i) {
    const int buf = int(i & 1);
    ok = ops.copy_in(i, buf) && ops.compute(i, buf) && ops.copy_out(i, buf);
  }
  if (ok) ok = ops.join();
  if (!ok) ops.drain();
  return ok ? GF_OK : GF_ERR_CUDA;
}

// The CUDA side's streams and events: two internal copy streams and the
// events that order the three stages, created by the call and released at
// its end (their resources go once the enqueued work completes).  A chain's
// pipe derives from this and says what each stage copies or computes.
struct CudaPipeBase : HostPipeOps {
  cudaStream_t s = nullptr;  // the caller's stream: the computes
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t ev_start = nullptr, ev_in[2] = {}, ev_comp[2] = {}, ev_out[2] = {};

  bool create() {
    bool ok = cudaStreamCreateWithFlags(&s_in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&s_out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&ev_start, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < 2; ++i)
      ok = cudaEventCreateWithFlags(&ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&ev_comp[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&ev_out[i], cudaEventDisableTiming) == cudaSuccess;
    return ok;
  }
  ~CudaPipeBase() override {
    for (int i = 0; i < 2; ++i) {
      if (ev_in[i]) cudaEventDestroy(ev_in[i]);
      if (ev_comp[i]) cudaEventDestroy(ev_comp[i]);
      if (ev_out[i]) cudaEventDestroy(ev_out[i]);
    }
    if (ev_start) cudaEventDestroy(ev_start);
    if (s_in) cudaStreamDestroy(s_in);
    if (s_out) cudaStreamDestroy(s_out);
  }
  // the copy streams start after everything already queued on `s`
  bool start() {
    return cudaEventRecord(ev_start, s) == cudaSuccess && cudaStreamWaitEvent(s_in, ev_start, 0) == cudaSuccess &&
           cudaStreamWaitEvent(s_out, ev_start, 0) == cudaSuccess;
  }
  bool copy_in_bytes(int buf, void* dev, const void* host, size_t bytes) {
    return cudaStreamWaitEvent(s_in, ev_comp[buf], 0) == cudaSuccess &&
           cudaMemcpyAsync(dev, host, bytes, cudaMemcpyHostToDevice, s_in) == cudaSuccess &&
           cudaEventRecord(ev_in[buf], s_in) == cudaSuccess;
  }
  bool compute_begin(int buf) {
    return cudaStreamWaitEvent(s, ev_in[buf], 0) == cudaSuccess && cudaStreamWaitEvent(s, ev_out[buf], 0) == cudaSuccess;
  }
  bool compute_end(int buf) { return cudaEventRecord(ev_comp[buf], s) == cudaSuccess; }
  bool copy_out_bytes(int buf, void* host, const void* dev, size_t bytes) {
    return cudaStreamWaitEvent(s_out, ev_comp[buf], 0) == cudaSuccess &&
           cudaMemcpyAsync(host, dev, bytes, cudaMemcpyDeviceToHost, s_out) == cudaSuccess &&
           cudaEventRecord(ev_out[buf], s_out) == cudaSuccess;
  }
  bool join() override {
    return cudaStreamWaitEvent(s, ev_out[0], 0) == cudaSuccess && cudaStreamWaitEvent(s, ev_out[1], 0) == cudaSuccess;
  }
  void drain() override {
    // blocks until the internal streams are idle (their copies wait on the
    // computes they depend on, so those finish too)
    if (s_in) cudaStreamSynchronize(s_in);
    if (s_out) cudaStreamSynchronize(s_out);
  }
};

}  // namespace gf
