// Host-buffer entry points of the per-sample chains: LayerNorm -> GELU ->
// dilated Conv1d -> +x (page Kimi-K2.6__l2_p5) and ConvTranspose3d -> Swish
// -> GroupNorm -> HardSwish (page Kimi-K2.6__l2_p60).  Both normalise within
// a sample (LayerNorm over [C, L], GroupNorm over a sample's channel groups),
// so a batch splits into chunks of whole samples that are computed by the
// device entry point one after another while the neighbouring chunks'
// copies run on the pipeline's internal streams (host_pipe.h).
#include <functional>

#include "host_common.h"
#include "host_pipe.h"

namespace gf {
namespace {

// Chunks of `chunk` samples of `in_item` input and `out_item` output bytes
// each; `run` computes one chunk from a device staging buffer into another
// on the caller's stream.
struct SampleHostPipe final : CudaPipeBase {
  const uint8_t* in_host = nullptr;
  uint8_t* out_host = nullptr;
  size_t in_item = 0, out_item = 0;
  int64_t items = 0, chunk = 1;
  uint8_t* in_dev[2] = {};
  uint8_t* out_dev[2] = {};
  std::function<gf_status(const void* in, void* out, int64_t n)> run;
  gf_status inner = GF_OK;  // the device entry point's status, when a compute failed

  int64_t n_of(int64_t i) const { return (items - i * chunk) < chunk ? (items - i * chunk) : chunk; }
  bool setup() override { return start(); }
  bool copy_in(int64_t i, int buf) override {
    return copy_in_bytes(buf, in_dev[buf], in_host + size_t(i * chunk) * in_item, size_t(n_of(i)) * in_item);
  }
  bool compute(int64_t i, int buf) override {
    return compute_begin(buf) && (inner = run(in_dev[buf], out_dev[buf], n_of(i))) == GF_OK && compute_end(buf);
  }
  bool copy_out(int64_t i, int buf) override {
    return copy_out_bytes(buf, out_host + size_t(i * chunk) * out_item, out_dev[buf], size_t(n_of(i)) * out_item);
  }
};

// Workspace of a per-sample pipeline: two input and two output staging
// buffers of `chunk` samples, then the device entry point's workspace for a
// chunk.
struct SampleWs {
  size_t in[2], out[2], inner, total;
};

SampleWs sample_ws(int64_t chunk, size_t in_item, size_t out_item, size_t inner_bytes) {
  SampleWs w{};
  size_t off = 0;
  for (int i = 0; i < 2; ++i) {
    w.in[i] = off;
    off += align_up(size_t(chunk) * in_item, 256);
  }
  for (int i = 0; i < 2; ++i) {
    w.out[i] = off;
    off += align_up(size_t(chunk) * out_item, 256);
  }
  w.inner = off;
  w.total = off + align_up(inner_bytes, 256);
  return w;
}

// Samples per chunk when the caller passes 0: eight chunks or fewer, so that
// the first chunk's copy-in and the last one's copy-out, which overlap
// nothing, are an eighth of the batch's copies.
int64_t default_chunk(int64_t n) { return n < 8 ? 1 : (n + 7) / 8; }

int64_t chunk_of(int64_t n, int64_t chunk_samples) {
  if (chunk_samples == 0) return default_chunk(n);
  return chunk_samples < n ? chunk_samples : n;
}

gf_status run_samples(SampleHostPipe& pipe, const SampleWs& w, void* workspace, void* stream) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  for (int i = 0; i < 2; ++i) {
    pipe.in_dev[i] = ws + w.in[i];
    pipe.out_dev[i] = ws + w.out[i];
  }
  pipe.s = static_cast<cudaStream_t>(stream);
  if (!pipe.create()) return GF_ERR_CUDA;  // nothing enqueued yet
  const gf_status st = run_host_pipeline(pipe, (pipe.items + pipe.chunk - 1) / pipe.chunk);
  // a compute that failed before any CUDA error reports the device entry
  // point's own status (its checks run on the first chunk)
  return st != GF_OK && pipe.inner != GF_OK ? pipe.inner : st;
}

int64_t convt_out_extent(int64_t n, int32_t k, int32_t stride, int32_t pad) { return (n - 1) * stride - 2 * pad + k; }

}  // namespace
}  // namespace gf

using namespace gf;

extern "C" {

size_t gf_ln_gelu_dconv1d_res_host_workspace_size(int64_t B, int64_t C, int64_t L, int32_t ksize, int32_t dilation,
                                                  int32_t mode, int64_t chunk_samples) {
  if (B <= 0 || C <= 0 || L <= 0 || chunk_samples < 0) return 0;
  const int64_t chunk = chunk_of(B, chunk_samples);
  const size_t inner = gf_ln_gelu_dconv1d_res_workspace_size(chunk, C, L, ksize, dilation, mode);
  if (inner == 0) return 0;
  const size_t item = size_t(C) * size_t(L) * 4;
  return sample_ws(chunk, item, item, inner).total;
}

gf_status gf_ln_gelu_dconv1d_res_host(const float* x_host, const float* ln_gamma, const float* ln_beta,
                                      const float* conv_w, const float* conv_b, float* out_host, int64_t B,
                                      int64_t C, int64_t L, int32_t ksize, int32_t dilation, int32_t padding,
                                      float eps, int32_t mode, int64_t chunk_samples, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  if (B < 0 || chunk_samples < 0) return GF_ERR_SHAPE;
  if (B == 0) return GF_OK;
  if (!x_host || !out_host || !workspace) return GF_ERR_NULL;
  const int64_t chunk = chunk_of(B, chunk_samples);
  const size_t inner = gf_ln_gelu_dconv1d_res_workspace_size(chunk, C, L, ksize, dilation, mode);
  if (inner == 0) return GF_ERR_SHAPE;
  if (!aligned16(workspace)) return GF_ERR_ALIGN;
  const size_t item = size_t(C) * size_t(L) * 4;
  const SampleWs w = sample_ws(chunk, item, item, inner);
  if (workspace_bytes < w.total) return GF_ERR_WORKSPACE;
  uint8_t* inner_ws = static_cast<uint8_t*>(workspace) + w.inner;
  SampleHostPipe pipe;
  pipe.in_host = reinterpret_cast<const uint8_t*>(x_host);
  pipe.out_host = reinterpret_cast<uint8_t*>(out_host);
  pipe.in_item = pipe.out_item = item;
  pipe.items = B;
  pipe.chunk = chunk;
  pipe.run = [=, &pipe](const void* in, void* out, int64_t n) {
    return gf_ln_gelu_dconv1d_res(static_cast<const float*>(in), ln_gamma, ln_beta, conv_w, conv_b,
                                  static_cast<float*>(out), n, C, L, ksize, dilation, padding, eps, mode, inner_ws,
                                  inner, pipe.s);
  };
  return run_samples(pipe, w, workspace, stream);
}

size_t gf_convt3d_swish_gn_hswish_host_workspace_size(int64_t N, int64_t Cin, int64_t Cout, int64_t D, int64_t H,
                                                      int64_t W, int32_t k, int32_t stride, int32_t pad,
                                                      int32_t groups, int64_t chunk_samples) {
  if (N <= 0 || chunk_samples < 0) return 0;
  const int64_t chunk = chunk_of(N, chunk_samples);
  const size_t inner = gf_convt3d_swish_gn_hswish_workspace_size(chunk, Cin, Cout, D, H, W, k, stride, pad, groups);
  if (inner == 0) return 0;
  const size_t in_item = size_t(Cin) * size_t(D * H * W) * 4;
  const size_t out_item = size_t(Cout) * size_t(convt_out_extent(D, k, stride, pad)) *
                          size_t(convt_out_extent(H, k, stride, pad)) * size_t(convt_out_extent(W, k, stride, pad)) * 4;
  return sample_ws(chunk, in_item, out_item, inner).total;
}

gf_status gf_convt3d_swish_gn_hswish_host(const float* x_host, const float* w, const float* b, const float* gamma,
                                          const float* beta, float* out_host, int64_t N, int64_t Cin, int64_t Cout,
                                          int64_t D, int64_t H, int64_t W, int32_t k, int32_t stride, int32_t pad,
                                          int32_t groups, float eps, int64_t chunk_samples, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  if (N < 0 || chunk_samples < 0) return GF_ERR_SHAPE;
  if (N == 0) return GF_OK;
  if (!x_host || !out_host || !workspace) return GF_ERR_NULL;
  const int64_t chunk = chunk_of(N, chunk_samples);
  const size_t inner = gf_convt3d_swish_gn_hswish_workspace_size(chunk, Cin, Cout, D, H, W, k, stride, pad, groups);
  if (inner == 0) return GF_ERR_SHAPE;
  if (!aligned16(workspace)) return GF_ERR_ALIGN;
  const size_t in_item = size_t(Cin) * size_t(D * H * W) * 4;
  const size_t out_item = size_t(Cout) * size_t(convt_out_extent(D, k, stride, pad)) *
                          size_t(convt_out_extent(H, k, stride, pad)) * size_t(convt_out_extent(W, k, stride, pad)) * 4;
  const SampleWs ws = sample_ws(chunk, in_item, out_item, inner);
  if (workspace_bytes < ws.total) return GF_ERR_WORKSPACE;
  uint8_t* inner_ws = static_cast<uint8_t*>(workspace) + ws.inner;
  SampleHostPipe pipe;
  pipe.in_host = reinterpret_cast<const uint8_t*>(x_host);
  pipe.out_host = reinterpret_cast<uint8_t*>(out_host);
  pipe.in_item = in_item;
  pipe.out_item = out_item;
  pipe.items = N;
  pipe.chunk = chunk;
  pipe.run = [=, &pipe](const void* in, void* out, int64_t n) {
    return gf_convt3d_swish_gn_hswish(static_cast<const float*>(in), w, b, gamma, beta, static_cast<float*>(out), n,
                                      Cin, Cout, D, H, W, k, stride, pad, groups, eps, inner_ws, inner, pipe.s);
  };
  return run_samples(pipe, ws, workspace, stream);
}

}  // extern "C"
