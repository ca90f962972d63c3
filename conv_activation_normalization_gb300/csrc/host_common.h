// Host-side helpers shared by the entry points: argument checks, device
// properties, TMA descriptor encoding and the device status word.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/gf.h"

namespace gf {

// Pointer checks --------------------------------------------------------
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Span {
  const void* p;
  size_t bytes;
};

// true when [a, a+na) and [b, b+nb) share a byte.
inline bool overlaps(Span a, Span b) {
  if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// GF_ERR_ALIAS when `out` overlaps any of the n inputs.
gf_status check_no_alias(Span out, const Span* ins, int n);

// Device ------------------------------------------------------------------
struct DeviceInfo {
  int device;
  int sm_count;
  int cc_major, cc_minor;
  int max_smem_optin;
};
// GF_OK and the current device's properties, or GF_ERR_CUDA /
// GF_ERR_UNSUPPORTED_ARCH (anything but sm_103).
gf_status current_device(DeviceInfo* info);

// Device address of the library's status word on the current device.
uint32_t* device_status_word();

// Unique id (cuCtxGetId) of the calling thread's current CUDA context.  A
// device address looked up with cudaGetSymbolAddress is cached together with
// this id and looked up again when the id changes (a context that was
// destroyed and recreated, e.g. by cudaDeviceReset, reloads the module).
gf_status current_context_id(unsigned long long* id);

gf_status cuda_status(cudaError_t e);

// TMA ---------------------------------------------------------------------
// Tiled tensor map of fp32 (elem_bytes 4) or bf16 (elem_bytes 2) data with
// 128-byte swizzle (or 64-byte, swizzle_bytes = 64) and zero fill out of
// bounds.  dims[0] is the contiguous dimension; strides are derived from a
// dense layout; box[0] * elem_bytes must equal the swizzle span.
gf_status make_tmap(CUtensorMap* map, const void* base, int elem_bytes, int rank, const uint64_t* dims,
                    const uint32_t* box, int swizzle_bytes = 128);

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Profiling: while gf_profile_begin() is active, every entry point records
// a pair of CUDA events on its stream around its dominant kernel.
void profile_mark_begin(cudaStream_t s);
void profile_mark_end(cudaStream_t s);

}  // namespace gf
