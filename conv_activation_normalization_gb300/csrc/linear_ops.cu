// The two Linear-based chains:
//   gf_linear_swish_bias_groupnorm   (page Kimi-K2.6__l2_p37)
//   gf_linear_lse_act                (page Kimi-K2.6__l2_p64)
// Both run a hi/lo split pre-pass on x and W, then one persistent tcgen05
// 3xTF32 GEMM whose epilogue does the rest of the chain on the accumulator
// tile in registers; the logsumexp chain adds a tiny per-row merge kernel.
#include <cmath>

#include "gemm_tc.cuh"
#include "host_common.h"
#include "kernels_common.cuh"

namespace gf {

// ------------------------------------------------------------- epilogues
// Linear -> Swish -> +bias -> GroupNorm on a 128 x BN accumulator tile; one
// thread owns one row, a group is 64 consecutive columns, so the group's mean
// and (two-pass, biased) variance are computed in the thread's registers.
struct EpiSwishBiasGN {
  struct Params {
    const float* b_lin;  // may be null
    const float* bias;
    const float* gamma;
    const float* beta;
    float* out;
    int M, N;
    float eps;
  };
  template <int BN>
  __device__ __forceinline__ static void apply(const Params& p, uint32_t taddr, const Tile& t, int row) {
    const int m = t.r0 + row;
    const bool valid = m < p.M;
#pragma unroll 1
    for (int g = 0; g < BN / 64; ++g) {
      const int n0 = t.n0 + g * 64;
      if (n0 >= p.N) break;  // uniform across the warp
      float v[64];
      tmem_load64(taddr + uint32_t(g * 64), v);
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < 64; j += 4) {
        const float4 bl = p.b_lin ? __ldg(reinterpret_cast<const float4*>(p.b_lin + n0 + j)) : make_float4(0, 0, 0, 0);
        const float4 bb = __ldg(reinterpret_cast<const float4*>(p.bias + n0 + j));
        v[j + 0] = swish(v[j + 0] + bl.x) + bb.x;
        v[j + 1] = swish(v[j + 1] + bl.y) + bb.y;
        v[j + 2] = swish(v[j + 2] + bl.z) + bb.z;
        v[j + 3] = swish(v[j + 3] + bl.w) + bb.w;
        sum += (v[j] + v[j + 1]) + (v[j + 2] + v[j + 3]);
      }
      const float mean = sum * (1.f / 64.f);
      float m2 = 0.f;
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const float d = v[j] - mean;
        m2 = fmaf(d, d, m2);
      }
      const float rstd = rsqrtf(m2 * (1.f / 64.f) + p.eps);
      float* orow = p.out + size_t(m) * size_t(p.N) + n0;
#pragma unroll
      for (int j = 0; j < 64; j += 4) {
        const float4 ga = __ldg(reinterpret_cast<const float4*>(p.gamma + n0 + j));
        const float4 be = __ldg(reinterpret_cast<const float4*>(p.beta + n0 + j));
        float4 o;
        o.x = fmaf((v[j + 0] - mean) * rstd, ga.x, be.x);
        o.y = fmaf((v[j + 1] - mean) * rstd, ga.y, be.y);
        o.z = fmaf((v[j + 2] - mean) * rstd, ga.z, be.z);
        o.w = fmaf((v[j + 3] - mean) * rstd, ga.w, be.w);
        if (valid) __stcs(reinterpret_cast<float4*>(orow + j), o);
      }
    }
  }
};

// Linear -> per-row (max, sum exp(y - max)) over the tile's BN columns,
// written as one float2 partial per (row, n-block).
struct EpiLSEPartial {
  struct Params {
    const float* b;  // may be null
    float2* part;    // [M][n_blocks]
    int M, N, n_blocks;
  };
  template <int BN>
  __device__ __forceinline__ static void apply(const Params& p, uint32_t taddr, const Tile& t, int row) {
    const int m = t.r0 + row;
    float mx = -INFINITY, s = 0.f;
#pragma unroll 1
    for (int g = 0; g < BN / 64; ++g) {
      const int n0 = t.n0 + g * 64;
      if (n0 >= p.N) break;  // uniform across the warp
      float v[64];
      tmem_load64(taddr + uint32_t(g * 64), v);
      float cm = -INFINITY;
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const int n = n0 + j;
        const float bj = (p.b && n < p.N) ? __ldg(p.b + n) : 0.f;
        v[j] = n < p.N ? v[j] + bj : -INFINITY;
        cm = fmaxf(cm, v[j]);
      }
      const float nm = fmaxf(mx, cm);
      s *= __expf(mx - nm);
#pragma unroll
      for (int j = 0; j < 64; ++j) s += __expf(v[j] - nm);
      mx = nm;
    }
    if (m < p.M) p.part[size_t(m) * p.n_blocks + t.nb] = make_float2(mx, s);
  }
};

// Plain Linear: out[m, n] = acc + b[n] (the contraction step alone).
struct EpiStore {
  struct Params {
    const float* b;  // may be null
    float* out;
    int M, N;
  };
  template <int BN>
  __device__ __forceinline__ static void apply(const Params& p, uint32_t taddr, const Tile& t, int row) {
    const int m = t.r0 + row;
    const bool valid = m < p.M;
#pragma unroll 1
    for (int g = 0; g < BN / 64; ++g) {
      const int n0 = t.n0 + g * 64;
      if (n0 >= p.N) break;  // uniform across the warp
      float v[64];
      tmem_load64(taddr + uint32_t(g * 64), v);
      float* orow = p.out + size_t(m) * size_t(p.N);
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const int n = n0 + j;
        if (valid && n < p.N) orow[n] = v[j] + (p.b ? __ldg(p.b + n) : 0.f);
      }
    }
  }
};

// ------------------------------------------------------- auxiliary kernels
// Merge a row's (max, sumexp) partials, then the scalar chain
// lse -> LeakyReLU -> LeakyReLU -> GELU -> GELU.  One warp per row.
__global__ void lse_merge_act_kernel(const float2* __restrict__ part, float* __restrict__ out, int M,
                                     int n_blocks, float slope) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (warp >= M) return;
  float mx = -INFINITY, s = 0.f;
  for (int i = lane; i < n_blocks; i += 32) {
    const float2 q = part[size_t(warp) * n_blocks + i];
    const float nm = fmaxf(mx, q.x);
    s = s * __expf(mx - nm) + q.y * __expf(q.x - nm);
    mx = nm;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, mx, o);
    const float os = __shfl_xor_sync(0xffffffffu, s, o);
    const float nm = fmaxf(mx, om);
    s = (mx == -INFINITY ? 0.f : s * __expf(mx - nm)) + (om == -INFINITY ? 0.f : os * __expf(om - nm));
    mx = nm;
  }
  if (lane == 0) {
    float a = mx + logf(s);
    a = a > 0.f ? a : slope * a;
    a = a > 0.f ? a : slope * a;
    a = gelu_erf(a);
    a = gelu_erf(a);
    out[warp] = a;
  }
}

// ------------------------------------------------------------ host side
namespace {

constexpr int kBNLinear = 256;

size_t planes_bytes(int64_t rows, int64_t K) { return align_up(size_t(2) * size_t(rows) * size_t(K) * 4, 256); }

gf_status check_linear_shape(int64_t M, int64_t K, int64_t N) {
  if (M < 1 || K < 4 || N < 1) return GF_ERR_SHAPE;
  if (K % 4) return GF_ERR_SHAPE;                        // TMA row stride must be 16-byte aligned
  if (M > (int64_t(1) << 31) - 256 || N > (int64_t(1) << 31) - 256 || K > (int64_t(1) << 31) - 64)
    return GF_ERR_SHAPE;                                 // TMA coordinates are int32
  return GF_OK;
}

template <class Epi>
gf_status launch_linear_gemm(const DeviceInfo& dev, const float* a_planes, const float* b_planes, int64_t M,
                             int64_t K, int64_t N, int m_fastest, const typename Epi::Params& ep,
                             cudaStream_t stream) {
  using Cfg = TileCfg<kBNLinear>;
  CUtensorMap ta, tb;
  const uint64_t da[3] = {uint64_t(K), uint64_t(M), 2};
  const uint32_t ba[3] = {kBK, kBM, 1};
  const uint64_t db[3] = {uint64_t(K), uint64_t(N), 2};
  const uint32_t bb[3] = {kBK, kBNLinear, 1};
  gf_status st = make_tmap_f32(&ta, a_planes, 3, da, ba);
  if (st != GF_OK) return st;
  st = make_tmap_f32(&tb, b_planes, 3, db, bb);
  if (st != GF_OK) return st;
  LinearSrc src;
  src.num_mb = int((M + kBM - 1) / kBM);
  src.num_nb = int((N + kBNLinear - 1) / kBNLinear);
  src.num_kb = int((K + kBK - 1) / kBK);
  src.bn = kBNLinear;
  src.m_fastest = m_fastest;
  const int64_t tiles = int64_t(src.num_mb) * src.num_nb;
  const int grid = int(tiles < dev.sm_count ? tiles : dev.sm_count);
  auto kern = gemm3xtf32_kernel<kBNLinear, LinearSrc, Epi>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
    return GF_ERR_CUDA;
  profile_mark_begin(stream);
  kern<<<grid, kGemmThreads, Cfg::SMEM_BYTES, stream>>>(ta, tb, src, ep, device_status_word());
  profile_mark_end(stream);
  return cuda_status(cudaGetLastError());
}

gf_status split_planes(const float* src, float* planes, int64_t rows, int64_t K, const DeviceInfo& dev,
                       cudaStream_t stream) {
  const size_t n = size_t(rows) * size_t(K);
  return launch_split_tf32(src, planes, planes + n, n, dev.sm_count, stream);
}

}  // namespace
}  // namespace gf

using namespace gf;

extern "C" {

size_t gf_linear_swish_bias_groupnorm_workspace_size(int64_t M, int64_t K, int64_t N, int32_t groups,
                                                     int32_t mode) {
  (void)groups;
  if (mode != GF_MODE_FP32_3XTF32 || check_linear_shape(M, K, N) != GF_OK) return 0;
  return planes_bytes(M, K) + planes_bytes(N, K);
}

gf_status gf_tf32_split(const float* src, float* planes, int64_t n, void* stream) {
  if (!src || !planes) return GF_ERR_NULL;
  if (n < 4 || n % 4) return GF_ERR_SHAPE;
  if (!aligned16(src) || !aligned16(planes)) return GF_ERR_ALIGN;
  const Span ins[] = {{src, size_t(n) * 4}};
  gf_status st = check_no_alias(Span{planes, size_t(n) * 8}, ins, 1);
  if (st != GF_OK) return st;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != GF_OK) return st;
  return launch_split_tf32(src, planes, planes + n, size_t(n), dev.sm_count, static_cast<cudaStream_t>(stream));
}

gf_status gf_linear_swish_bias_groupnorm_planes(const float* x_planes, const float* W_planes, const float* b_lin,
                                                const float* bias, const float* gamma, const float* beta, float* out,
                                                int64_t M, int64_t K, int64_t N, int32_t groups, float eps,
                                                void* stream) {
  if (!x_planes || !W_planes || !bias || !gamma || !beta || !out) return GF_ERR_NULL;
  gf_status st = check_linear_shape(M, K, N);
  if (st != GF_OK) return st;
  if (groups < 1 || N % groups != 0 || N / groups != 64) return GF_ERR_SHAPE;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return GF_ERR_SHAPE;
  if (!aligned16(x_planes) || !aligned16(W_planes) || !aligned16(bias) || !aligned16(gamma) || !aligned16(beta) ||
      !aligned16(out) || (b_lin && !aligned16(b_lin)))
    return GF_ERR_ALIGN;
  const Span ins[] = {{x_planes, size_t(M) * K * 8}, {W_planes, size_t(N) * K * 8}, {b_lin, size_t(N) * 4},
                      {bias, size_t(N) * 4},         {gamma, size_t(N) * 4},         {beta, size_t(N) * 4}};
  st = check_no_alias(Span{out, size_t(M) * N * 4}, ins, 6);
  if (st != GF_OK) return st;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != GF_OK) return st;
  EpiSwishBiasGN::Params ep{b_lin, bias, gamma, beta, out, int(M), int(N), eps};
  // n-blocks fastest: the CTAs in flight share a few m-blocks of x, while all
  // of W (N x K planes) stays resident in L2.
  return launch_linear_gemm<EpiSwishBiasGN>(dev, x_planes, W_planes, M, K, N, /*m_fastest=*/0, ep,
                                            static_cast<cudaStream_t>(stream));
}

gf_status gf_linear_swish_bias_groupnorm(const float* x, const float* W, const float* b_lin, const float* bias,
                                         const float* gamma, const float* beta, float* out, int64_t M,
                                         int64_t K, int64_t N, int32_t groups, float eps, int32_t mode,
                                         void* workspace, size_t workspace_bytes, void* stream) {
  if (!x || !W || !bias || !gamma || !beta || !out) return GF_ERR_NULL;
  if (mode != GF_MODE_FP32_3XTF32) return GF_ERR_MODE;
  gf_status st = check_linear_shape(M, K, N);
  if (st != GF_OK) return st;
  if (groups < 1 || N % groups != 0 || N / groups != 64) return GF_ERR_SHAPE;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return GF_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(W) || !aligned16(bias) || !aligned16(gamma) || !aligned16(beta) ||
      !aligned16(out) || (b_lin && !aligned16(b_lin)) || !aligned16(workspace))
    return GF_ERR_ALIGN;
  const size_t need = gf_linear_swish_bias_groupnorm_workspace_size(M, K, N, groups, mode);
  if (!workspace) return GF_ERR_NULL;
  if (workspace_bytes < need) return GF_ERR_WORKSPACE;
  const Span ins[] = {{x, size_t(M) * K * 4}, {W, size_t(N) * K * 4}, {b_lin, size_t(N) * 4},
                      {bias, size_t(N) * 4},  {gamma, size_t(N) * 4}, {beta, size_t(N) * 4},
                      {workspace, need}};
  st = check_no_alias(Span{out, size_t(M) * N * 4}, ins, 7);
  if (st != GF_OK) return st;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != GF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  float* a_planes = static_cast<float*>(workspace);
  float* b_planes = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + planes_bytes(M, K));
  if ((st = split_planes(x, a_planes, M, K, dev, s)) != GF_OK) return st;
  if ((st = split_planes(W, b_planes, N, K, dev, s)) != GF_OK) return st;
  return gf_linear_swish_bias_groupnorm_planes(a_planes, b_planes, b_lin, bias, gamma, beta, out, M, K, N, groups,
                                               eps, stream);
}

size_t gf_linear_workspace_size(int64_t M, int64_t K, int64_t N, int32_t mode) {
  if (mode != GF_MODE_FP32_3XTF32 || check_linear_shape(M, K, N) != GF_OK) return 0;
  return planes_bytes(M, K) + planes_bytes(N, K);
}

gf_status gf_linear(const float* x, const float* W, const float* b, float* out, int64_t M, int64_t K, int64_t N,
                    int32_t mode, void* workspace, size_t workspace_bytes, void* stream) {
  if (!x || !W || !out) return GF_ERR_NULL;
  if (mode != GF_MODE_FP32_3XTF32) return GF_ERR_MODE;
  gf_status st = check_linear_shape(M, K, N);
  if (st != GF_OK) return st;
  if (!aligned16(x) || !aligned16(W) || !aligned16(out) || (b && !aligned16(b)) || !aligned16(workspace))
    return GF_ERR_ALIGN;
  const size_t need = gf_linear_workspace_size(M, K, N, mode);
  if (!workspace) return GF_ERR_NULL;
  if (workspace_bytes < need) return GF_ERR_WORKSPACE;
  const Span ins[] = {{x, size_t(M) * K * 4}, {W, size_t(N) * K * 4}, {b, size_t(N) * 4}, {workspace, need}};
  st = check_no_alias(Span{out, size_t(M) * N * 4}, ins, 4);
  if (st != GF_OK) return st;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != GF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* a_planes = static_cast<float*>(workspace);
  float* b_planes = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + planes_bytes(M, K));
  if ((st = split_planes(x, a_planes, M, K, dev, s)) != GF_OK) return st;
  if ((st = split_planes(W, b_planes, N, K, dev, s)) != GF_OK) return st;
  EpiStore::Params ep{b, out, int(M), int(N)};
  return launch_linear_gemm<EpiStore>(dev, a_planes, b_planes, M, K, N, /*m_fastest=*/0, ep, s);
}

size_t gf_linear_lse_act_workspace_size(int64_t M, int64_t K, int64_t N, int32_t mode) {
  if (mode != GF_MODE_FP32_3XTF32 || check_linear_shape(M, K, N) != GF_OK) return 0;
  const int64_t nb = (N + kBNLinear - 1) / kBNLinear;
  return planes_bytes(M, K) + planes_bytes(N, K) + align_up(size_t(M) * nb * sizeof(float2), 256);
}

gf_status gf_linear_lse_act(const float* x, const float* W, const float* b, float* out, int64_t M, int64_t K,
                            int64_t N, float negative_slope, int32_t mode, void* workspace,
                            size_t workspace_bytes, void* stream) {
  if (!x || !W || !out) return GF_ERR_NULL;
  if (mode != GF_MODE_FP32_3XTF32) return GF_ERR_MODE;
  gf_status st = check_linear_shape(M, K, N);
  if (st != GF_OK) return st;
  if (!std::isfinite(negative_slope)) return GF_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(W) || !aligned16(out) || (b && !aligned16(b)) || !aligned16(workspace))
    return GF_ERR_ALIGN;
  const size_t need = gf_linear_lse_act_workspace_size(M, K, N, mode);
  if (!workspace) return GF_ERR_NULL;
  if (workspace_bytes < need) return GF_ERR_WORKSPACE;
  const Span ins[] = {{x, size_t(M) * K * 4}, {W, size_t(N) * K * 4}, {b, size_t(N) * 4}, {workspace, need}};
  st = check_no_alias(Span{out, size_t(M) * 4}, ins, 4);
  if (st != GF_OK) return st;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != GF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* a_planes = reinterpret_cast<float*>(ws);
  float* b_planes = reinterpret_cast<float*>(ws + planes_bytes(M, K));
  float2* part = reinterpret_cast<float2*>(ws + planes_bytes(M, K) + planes_bytes(N, K));
  const int nb = int((N + kBNLinear - 1) / kBNLinear);
  if ((st = split_planes(x, a_planes, M, K, dev, s)) != GF_OK) return st;
  if ((st = split_planes(W, b_planes, N, K, dev, s)) != GF_OK) return st;
  EpiLSEPartial::Params ep{b, part, int(M), int(N), nb};
  // m-blocks fastest: the CTAs in flight share n-blocks, so each W tile is
  // fetched from HBM once and reused by every m-block from L2.
  if ((st = launch_linear_gemm<EpiLSEPartial>(dev, a_planes, b_planes, M, K, N, /*m_fastest=*/1, ep, s)) != GF_OK)
    return st;
  const int threads = 256;
  const int blocks = int((M * 32 + threads - 1) / threads);
  lse_merge_act_kernel<<<blocks, threads, 0, s>>>(part, out, int(M), nb, negative_slope);
  return cuda_status(cudaGetLastError());
}

}  // extern "C"
