// Small device functions and the hi/lo split pre-pass shared by the
// tensor-core paths.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/gf.h"

namespace gf {

// Swish / SiLU: v * sigmoid(v) = v / (1 + e^-v).  For v < about -88, e^-v is
// inf and the quotient is the correct limit -0.
__device__ __forceinline__ float swish(float v) { return __fdividef(v, 1.0f + __expf(-v)); }

// Packed pair arithmetic: one f32x2 instruction (round to nearest) works on
// both lanes of a float2.
__device__ __forceinline__ unsigned long long f2_as_u64(float2 a) { return *reinterpret_cast<unsigned long long*>(&a); }
__device__ __forceinline__ float2 u64_as_f2(unsigned long long a) { return *reinterpret_cast<float2*>(&a); }

// d = a * b + c on both lanes of a pair (fma.rn.f32x2).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(f2_as_u64(a)), "l"(f2_as_u64(b)), "l"(f2_as_u64(c)));
  return u64_as_f2(d);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_as_u64(a)), "l"(f2_as_u64(b)));
  return u64_as_f2(d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_as_u64(a)), "l"(f2_as_u64(b)));
  return u64_as_f2(d);
}

// The special-function unit's 2^t and 1/d (ex2.approx / rcp.approx, denormal
// results flushed to zero).
__device__ __forceinline__ float ex2_approx(float t) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
  return r;
}
__device__ __forceinline__ float rcp_approx(float d) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
  return r;
}

// Swish of a pair, v * 1 / (1 + 2^(-v log2 e)), with the multiplies and the
// add packed.  Same limits as swish(): e^-v = inf gives 1/inf = 0 and -0.
__device__ __forceinline__ float2 swish2(float2 v) {
  constexpr float kNegLog2e = -1.4426950408889634f;
  const float2 t = mul2(v, make_float2(kNegLog2e, kNegLog2e));
  const float2 d = add2(make_float2(ex2_approx(t.x), ex2_approx(t.y)), make_float2(1.f, 1.f));
  return mul2(v, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
}

// Exact GELU v * Phi(v) = 0.5 v (1 + erf(v / sqrt 2)), with CUDA's erff.
__device__ __forceinline__ float gelu_erf(float v) { return 0.5f * v * (1.0f + erff(v * 0.70710678118654752f)); }
// GELU's tanh approximation 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))),
// with CUDA's tanhf.
__device__ __forceinline__ float gelu_tanh(float v) {
  return 0.5f * v * (1.0f + tanhf(0.79788456080286536f * fmaf(0.044715f * v, v * v, v)));
}

// TF32 split: hi keeps the sign, exponent and top 10 mantissa bits (exactly a
// TF32 value), lo = v - hi is exact in fp32.
__device__ __forceinline__ float tf32_hi(float v) { return __uint_as_float(__float_as_uint(v) & 0xFFFFE000u); }

static __global__ void split_tf32_kernel(const float4* __restrict__ src, float4* __restrict__ hi,
                                         float4* __restrict__ lo, size_t n4) {
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += size_t(gridDim.x) * blockDim.x) {
    const float4 v = __ldcs(src + i);
    float4 h, l;
    h.x = tf32_hi(v.x);
    h.y = tf32_hi(v.y);
    h.z = tf32_hi(v.z);
    h.w = tf32_hi(v.w);
    l.x = v.x - h.x;
    l.y = v.y - h.y;
    l.z = v.z - h.z;
    l.w = v.w - h.w;
    hi[i] = h;
    lo[i] = l;
  }
}

// lo = v - tf32_hi(v) only (the tensor core reads the raw value as hi).
static __global__ void split_lo_tf32_kernel(const float4* __restrict__ src, float4* __restrict__ lo, size_t n4) {
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += size_t(gridDim.x) * blockDim.x) {
    const float4 v = __ldcs(src + i);
    lo[i] = make_float4(v.x - tf32_hi(v.x), v.y - tf32_hi(v.y), v.z - tf32_hi(v.z), v.w - tf32_hi(v.w));
  }
}

// BF16 split: hi = bf16(v) (round to nearest even), lo = bf16(v - hi); with
// lo == nullptr only hi is written.
struct Bf16x4 {
  __nv_bfloat162 a, b;
};
__device__ __forceinline__ void bf16_split4(float4 v, Bf16x4& h, Bf16x4& l) {
  h.a = __floats2bfloat162_rn(v.x, v.y);
  h.b = __floats2bfloat162_rn(v.z, v.w);
  const float2 ha = __bfloat1622float2(h.a), hb = __bfloat1622float2(h.b);
  l.a = __floats2bfloat162_rn(v.x - ha.x, v.y - ha.y);
  l.b = __floats2bfloat162_rn(v.z - hb.x, v.w - hb.y);
}

static __global__ void split_bf16_kernel(const float4* __restrict__ src, Bf16x4* __restrict__ hi,
                                         Bf16x4* __restrict__ lo, size_t n4) {
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += size_t(gridDim.x) * blockDim.x) {
    Bf16x4 h, l;
    bf16_split4(__ldcs(src + i), h, l);
    hi[i] = h;
    if (lo) lo[i] = l;
  }
}

static inline int split_blocks(size_t n4, int sm_count) {
  const size_t blocks = (n4 + 255) / 256;
  const size_t cap = size_t(sm_count) * 8;
  return int(blocks > cap ? cap : blocks);
}

// n must be a multiple of 4; src and the fp32 planes 16-byte aligned, the
// bf16 planes 8-byte aligned.
static inline gf_status launch_split_lo_tf32(const float* src, float* lo, size_t n, int sm_count,
                                             cudaStream_t stream) {
  const size_t n4 = n / 4;
  if (n4 == 0) return GF_OK;
  split_lo_tf32_kernel<<<split_blocks(n4, sm_count), 256, 0, stream>>>(reinterpret_cast<const float4*>(src),
                                                                       reinterpret_cast<float4*>(lo), n4);
  return cudaGetLastError() == cudaSuccess ? GF_OK : GF_ERR_CUDA;
}

static inline gf_status launch_split_bf16(const float* src, void* hi, void* lo, size_t n, int sm_count,
                                          cudaStream_t stream) {
  const size_t n4 = n / 4;
  if (n4 == 0) return GF_OK;
  split_bf16_kernel<<<split_blocks(n4, sm_count), 256, 0, stream>>>(
      reinterpret_cast<const float4*>(src), static_cast<Bf16x4*>(hi), static_cast<Bf16x4*>(lo), n4);
  return cudaGetLastError() == cudaSuccess ? GF_OK : GF_ERR_CUDA;
}

// n must be a multiple of 4 and all pointers 16-byte aligned.
static inline gf_status launch_split_tf32(const float* src, float* hi, float* lo, size_t n, int sm_count,
                                          cudaStream_t stream) {
  const size_t n4 = n / 4;
  if (n4 == 0) return GF_OK;
  const int threads = 256;
  size_t blocks = (n4 + threads - 1) / threads;
  const size_t cap = size_t(sm_count) * 8;
  if (blocks > cap) blocks = cap;
  split_tf32_kernel<<<unsigned(blocks), threads, 0, stream>>>(reinterpret_cast<const float4*>(src),
                                                             reinterpret_cast<float4*>(hi),
                                                             reinterpret_cast<float4*>(lo), n4);
  return cudaGetLastError() == cudaSuccess ? GF_OK : GF_ERR_CUDA;
}

}  // namespace gf
