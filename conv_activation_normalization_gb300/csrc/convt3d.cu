// ConvTranspose3d(k 3, stride 2, pad 1) -> Swish -> GroupNorm -> HardSwish
//                                               (page Kimi-K2.6__l2_p60)
//
// This file holds the entry points (which send every other kernel size,
// stride, padding, channel count or group count to convt3d_general.cu) and
// the CUDA-core kernels of the pages' configuration for 4 < Cin <= 8 and the
// no-workspace entry point; Cin <= 4 runs on the tensor cores
// (convt3d_tc.cuh, convt3d_fused.cuh).
//
// Sub-pixel (phase) form of the transposed convolution.  Output index o
// along one dimension is o = 2 i - 1 + k; splitting o into a cell q and a
// phase p (o = 2q + p):
//   p = 0  gets one tap:  (i = q,     k = 1)
//   p = 1  gets two taps: (i = q + 1, k = 0) and (i = q, k = 2)
// so the 2x2x2 outputs of cell (qd, qh, qw) read only the 2x2x2 inputs at
// q..q+1 and every one of the 27 taps feeds exactly one phase: no zero
// (inserted) taps are multiplied and there are no per-output branches.  The
// last cell along a dimension (q = I - 1) has only its p = 0 output; its
// missing input q + 1 is read as 0 and its p = 1 output is not kept.
//
// GroupNorm needs the statistics of the whole (sample, group) before any
// output can be written, and the 1 GB output does not fit on chip, so:
//   pass 1  conv + bias + Swish, per-block (sum, sum of squares) per group
//           (fp32 within a warp, fp64 across warps) -- nothing is stored;
//   finalize per (sample, channel): fp64 merge -> A = gamma * rstd,
//           B = beta - mean * A;
//   pass 2  recompute conv + bias + Swish, h = A s + B, HardSwish, store.
// Each thread owns one cell and one group of 4 output channels at a time
// (Cout = 16 with 4 groups, so a group is 4 channels): 32 accumulators; the
// weights sit in shared memory as [ci][tap][co], read as float4 broadcasts.
#include <cmath>
#include <mutex>

#include "convt3d_fused.cuh"
#include "convt3d_general.h"
#include "convt3d_tc.cuh"
#include "host_common.h"
#include "kernels_common.cuh"

namespace gf {

constexpr int kCT_COUT = 16;
constexpr int kCT_G = 4;
constexpr int kCT_TX = 32, kCT_TY = 8;  // cells per block along w and h

// The 2x2x2 inputs of a cell, each held twice ((v, v) pairs) so the packed
// f32x2 FMAs below can multiply one input by the weights of two channels.
template <int CIN>
struct CellInputs {
  float2 v[CIN][2][2][2];
};

template <int CIN>
__device__ __forceinline__ void load_cell(CellInputs<CIN>& in, const float* __restrict__ xn, int D, int H, int W,
                                          int qd, int qh, int qw) {
#pragma unroll
  for (int ci = 0; ci < CIN; ++ci)
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int d = qd + a, h = qh + b, w = qw + c;
          float v = 0.f;
          if (d < D && h < H && w < W) v = __ldg(xn + ((size_t(ci) * D + d) * H + h) * W + w);
          in.v[ci][a][b][c] = make_float2(v, v);
        }
}

// Accumulators of one cell for the 4 channels of group cg, as channel pairs:
// a01[phase] = (channel 0, channel 1), a23[phase] = (channel 2, channel 3),
// phase = pd*4 + ph*2 + pw.  ws = smem weights [CIN][27][16], bias4 = conv
// bias of the 4 channels.
template <int CIN>
__device__ __forceinline__ void conv_cell(const CellInputs<CIN>& in, const float* __restrict__ ws, int cg,
                                          float4 bias4, float2 (&a01)[8], float2 (&a23)[8]) {
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    a01[p] = make_float2(bias4.x, bias4.y);
    a23[p] = make_float2(bias4.z, bias4.w);
  }
#pragma unroll
  for (int ci = 0; ci < CIN; ++ci)
#pragma unroll
    for (int kd = 0; kd < 3; ++kd)
#pragma unroll
      for (int kh = 0; kh < 3; ++kh)
#pragma unroll
        for (int kw = 0; kw < 3; ++kw) {
          // tap k -> (phase p, input offset a): k=1 -> (0, 0); k=0 -> (1, 1); k=2 -> (1, 0)
          const int pd = kd == 1 ? 0 : 1, ad = kd == 0 ? 1 : 0;
          const int ph = kh == 1 ? 0 : 1, ah = kh == 0 ? 1 : 0;
          const int pw = kw == 1 ? 0 : 1, aw = kw == 0 ? 1 : 0;
          const int phase = pd * 4 + ph * 2 + pw;
          const float4 w4 = *reinterpret_cast<const float4*>(ws + (ci * 27 + (kd * 3 + kh) * 3 + kw) * 16 + cg * 4);
          const float2 xv = in.v[ci][ad][ah][aw];
          a01[phase] = fma2(xv, make_float2(w4.x, w4.y), a01[phase]);
          a23[phase] = fma2(xv, make_float2(w4.z, w4.w), a23[phase]);
        }
}

// Copy w[ci][co][27] to smem as [ci][27][co].
template <int CIN>
__device__ __forceinline__ void stage_weights(float* ws, const float* __restrict__ w) {
  for (int i = threadIdx.x + threadIdx.y * blockDim.x; i < CIN * 27 * kCT_COUT; i += blockDim.x * blockDim.y) {
    const int co = i % kCT_COUT;
    const int tap = (i / kCT_COUT) % 27;
    const int ci = i / (kCT_COUT * 27);
    ws[i] = __ldg(w + (size_t(ci) * kCT_COUT + co) * 27 + tap);
  }
}

__device__ __forceinline__ uint32_t phase_mask(int qd, int qh, int qw, int D, int H, int W) {
  // bit `phase` set when the output (2qd+pd, 2qh+ph, 2qw+pw) exists
  uint32_t m = 0;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const int pd = p >> 2, ph = (p >> 1) & 1, pw = p & 1;
    const bool ok = (pd == 0 || qd < D - 1) && (ph == 0 || qh < H - 1) && (pw == 0 || qw < W - 1);
    m |= uint32_t(ok) << p;
  }
  return m;
}

// grid (ceil(W/32), ceil(H/8), D * N), block (32, 8).
// part: [N][G][P][2] doubles, P = blocks per sample.
template <int CIN>
__global__ void __launch_bounds__(256, CIN <= 4 ? 3 : 2) convt3d_stats_kernel(const float* __restrict__ x, const float* __restrict__ w,
                                                            const float* __restrict__ bias, double* __restrict__ part,
                                                            int D, int H, int W) {
  __shared__ __align__(16) float ws[CIN * 27 * kCT_COUT];
  __shared__ double red[8][kCT_G][2];
  stage_weights<CIN>(ws, w);
  __syncthreads();
  const int n = blockIdx.z / D, qd = blockIdx.z % D;
  const int qh = blockIdx.y * kCT_TY + threadIdx.y, qw = blockIdx.x * kCT_TX + threadIdx.x;
  const bool cell_ok = qh < H && qw < W;
  CellInputs<CIN> in;
  load_cell<CIN>(in, x + size_t(n) * CIN * D * H * W, D, H, W, qd, qh, qw);
  const uint32_t pm = cell_ok ? phase_mask(qd, qh, qw, D, H, W) : 0u;
  const int lane = threadIdx.x, wid = threadIdx.y;
#pragma unroll 1
  for (int cg = 0; cg < kCT_G; ++cg) {
    const float4 b4 = bias ? __ldg(reinterpret_cast<const float4*>(bias) + cg) : make_float4(0, 0, 0, 0);
    float2 a01[8], a23[8];
    conv_cell<CIN>(in, ws, cg, b4, a01, a23);
    float a = 0.f, q = 0.f;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      if ((pm >> p) & 1u) {
        const float s0 = swish(a01[p].x), s1 = swish(a01[p].y), s2 = swish(a23[p].x), s3 = swish(a23[p].y);
        a += (s0 + s1) + (s2 + s3);
        q = fmaf(s0, s0, fmaf(s1, s1, fmaf(s2, s2, fmaf(s3, s3, q))));
      }
    }
    // warp reduction in fp32; the 8 warps are summed in fp64 below
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a += __shfl_xor_sync(0xffffffffu, a, o);
      q += __shfl_xor_sync(0xffffffffu, q, o);
    }
    if (lane == 0) {
      red[wid][cg][0] = a;
      red[wid][cg][1] = q;
    }
  }
  __syncthreads();
  if (wid == 0 && lane < 2 * kCT_G) {
    const int cg = lane >> 1, k = lane & 1;
    double t = 0.0;
#pragma unroll
    for (int i = 0; i < 8; ++i) t += red[i][cg][k];
    const int P = gridDim.x * gridDim.y * D;
    const int blk = (qd * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    part[((size_t(n) * kCT_G + cg) * P + blk) * 2 + k] = t;
  }
}

// grid N, block 64: merge the partials of each (n, group) -> per-channel
// affine A = gamma * rstd, B = beta - mean * A (coef[n][co] = (A, B)).
__global__ void convt3d_finalize_kernel(const double* __restrict__ part, const float* __restrict__ gamma,
                                        const float* __restrict__ beta, float2* __restrict__ coef, int P,
                                        double count, float eps) {
  __shared__ double acc[kCT_G][2][16];
  const int n = blockIdx.x;
  const int t = threadIdx.x;            // 64 threads: (group, k, slice)
  const int g = t / 16, sl = t % 16;
  double s = 0.0, q = 0.0;
  for (int i = sl; i < P; i += 16) {
    const double* p = part + ((size_t(n) * kCT_G + g) * P + i) * 2;
    s += p[0];
    q += p[1];
  }
  acc[g][0][sl] = s;
  acc[g][1][sl] = q;
  __syncthreads();
  if (t < kCT_COUT) {
    const int gg = t / (kCT_COUT / kCT_G);
    double S = 0.0, Q = 0.0;
    for (int i = 0; i < 16; ++i) {
      S += acc[gg][0][i];
      Q += acc[gg][1][i];
    }
    const double mean = S / count;
    const double var = fmax(Q / count - mean * mean, 0.0);
    const double rstd = 1.0 / sqrt(var + double(eps));
    const double A = double(gamma[t]) * rstd;
    coef[size_t(n) * kCT_COUT + t] = make_float2(float(A), float(double(beta[t]) - mean * A));
  }
}

// Same merge for float2 partials (the tensor-core path writes one per tile and
// epilogue warp): grid (N, groups), block 256; fp64 sums.
__global__ void __launch_bounds__(256) convt3d_finalize_f2_kernel(const float2* __restrict__ part,
                                                                  const float* __restrict__ gamma,
                                                                  const float* __restrict__ beta,
                                                                  float4* __restrict__ coef, int P, double count,
                                                                  float eps) {
  __shared__ double red[8][2];
  const int n = blockIdx.x, g = blockIdx.y;
  const float2* pg = part + (size_t(n) * kCT_G + g) * P;
  double s = 0.0, q = 0.0;
  for (int i = threadIdx.x; i < P; i += blockDim.x) {
    const float2 v = __ldg(pg + i);
    s += v.x;
    q += v.y;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, o);
    q += __shfl_xor_sync(0xffffffffu, q, o);
  }
  if ((threadIdx.x & 31) == 0) {
    red[threadIdx.x >> 5][0] = s;
    red[threadIdx.x >> 5][1] = q;
  }
  __syncthreads();
  if (threadIdx.x < kCT_COUT / kCT_G) {
    double S = 0.0, Q = 0.0;
    for (int w = 0; w < 8; ++w) {
      S += red[w][0];
      Q += red[w][1];
    }
    const double mean = S / count;
    const double var = fmax(Q / count - mean * mean, 0.0);
    const double rstd = 1.0 / sqrt(var + double(eps));
    const int c = g * (kCT_COUT / kCT_G) + threadIdx.x;
    const double A = double(gamma[c]) * rstd;
    const float Af = float(A), Bf = float(double(beta[c]) - mean * A);
    coef[size_t(n) * kCT_COUT + c] = make_float4(Af, Af, Bf, Bf);
  }
}

// HardSwish h * clamp(h + 3, 0, 6) / 6 written as h * sat(h / 6 + 1/2): one
// saturating FMA and one multiply.
__device__ __forceinline__ float hardswish(float h) { return h * __saturatef(fmaf(h, 1.f / 6.f, 0.5f)); }

// GroupNorm affine of Swish: A * swish(y) + B.
__device__ __forceinline__ float gn_swish(float y, float A, float B) { return fmaf(A, swish(y), B); }

template <int CIN>
__global__ void __launch_bounds__(256, CIN <= 4 ? 3 : 2) convt3d_apply_kernel(const float* __restrict__ x, const float* __restrict__ w,
                                                            const float* __restrict__ bias,
                                                            const float2* __restrict__ coef, float* __restrict__ out,
                                                            int D, int H, int W) {
  __shared__ __align__(16) float ws[CIN * 27 * kCT_COUT];
  stage_weights<CIN>(ws, w);
  __syncthreads();
  const int n = blockIdx.z / D, qd = blockIdx.z % D;
  const int qh = blockIdx.y * kCT_TY + threadIdx.y, qw = blockIdx.x * kCT_TX + threadIdx.x;
  const bool cell_ok = qh < H && qw < W;
  const int OD = 2 * D - 1, OH = 2 * H - 1, OW = 2 * W - 1;
  const int plane = OD * OH * OW;  // < 2^31 (checked on the host)
  CellInputs<CIN> in;
  load_cell<CIN>(in, x + size_t(n) * CIN * D * H * W, D, H, W, qd, qh, qw);
  const uint32_t pm = cell_ok ? phase_mask(qd, qh, qw, D, H, W) : 0u;
  // in-plane offset of the cell's first output (clamped for cells outside the
  // grid, whose outputs are masked off anyway)
  const int cell_off = (2 * qd * OH + 2 * min(qh, H - 1)) * OW + 2 * min(qw, W - 1);
  const int OHW = OH * OW;
#pragma unroll 1
  for (int cg = 0; cg < kCT_G; ++cg) {
    const float4 b4 = bias ? __ldg(reinterpret_cast<const float4*>(bias) + cg) : make_float4(0, 0, 0, 0);
    float2 a01[8], a23[8];
    conv_cell<CIN>(in, ws, cg, b4, a01, a23);
    const float4 ab01 = __ldg(reinterpret_cast<const float4*>(coef + size_t(n) * kCT_COUT + cg * 4));
    const float4 ab23 = __ldg(reinterpret_cast<const float4*>(coef + size_t(n) * kCT_COUT + cg * 4 + 2));
    float* o0 = out + (size_t(n) * kCT_COUT + cg * 4) * size_t(plane);
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      if ((pm >> p) & 1u) {
        const int po = cell_off + (p >> 2) * OHW + ((p >> 1) & 1) * OW + (p & 1);
        __stcs(o0 + po, hardswish(gn_swish(a01[p].x, ab01.x, ab01.y)));
        __stcs(o0 + plane + po, hardswish(gn_swish(a01[p].y, ab01.z, ab01.w)));
        __stcs(o0 + 2 * size_t(plane) + po, hardswish(gn_swish(a23[p].x, ab23.x, ab23.y)));
        __stcs(o0 + 3 * size_t(plane) + po, hardswish(gn_swish(a23[p].y, ab23.z, ab23.w)));
      }
    }
  }
}

namespace {
struct CtWs {
  size_t part, coef, total;
  int P;
};

CtWs ct_ws(int64_t N, int64_t D, int64_t H, int64_t W) {
  CtWs c{};
  c.P = int(((W + kCT_TX - 1) / kCT_TX) * ((H + kCT_TY - 1) / kCT_TY) * D);
  c.part = 0;
  c.coef = align_up(size_t(N) * kCT_G * c.P * 2 * sizeof(double), 256);
  c.total = c.coef + align_up(size_t(N) * kCT_COUT * sizeof(float4), 256);
  return c;
}

gf_status check_ct_shape(int64_t N, int64_t Cin, int64_t Cout, int64_t D, int64_t H, int64_t W, int32_t k,
                         int32_t stride, int32_t pad, int32_t groups) {
  if (k != 3 || stride != 2 || pad != 1) return GF_ERR_SHAPE;
  if (Cout != kCT_COUT || groups != kCT_G) return GF_ERR_SHAPE;
  if (Cin < 1 || Cin > 8 || N < 1 || D < 1 || H < 1 || W < 1) return GF_ERR_SHAPE;
  if (D * N > 65535 || (H + kCT_TY - 1) / kCT_TY > 65535 || W > (int64_t(1) << 20)) return GF_ERR_SHAPE;
  if (D > (1 << 20) || H > (1 << 20)) return GF_ERR_SHAPE;
  if ((2 * D - 1) * (2 * H - 1) * (2 * W - 1) >= (int64_t(1) << 31)) return GF_ERR_SHAPE;  // 32-bit in-plane offsets
  return GF_OK;
}

template <int CIN>
void launch_ct(const float* x, const float* w, const float* b, double* part, const float* gamma, const float* beta,
               float2* coef, float* out, int N, int D, int H, int W, int P, float eps, cudaStream_t s) {
  const dim3 grid((W + kCT_TX - 1) / kCT_TX, (H + kCT_TY - 1) / kCT_TY, D * N), block(kCT_TX, kCT_TY);
  convt3d_stats_kernel<CIN><<<grid, block, 0, s>>>(x, w, b, part, D, H, W);
  const double count = double(kCT_COUT / kCT_G) * double(2 * D - 1) * double(2 * H - 1) * double(2 * W - 1);
  convt3d_finalize_kernel<<<N, 64, 0, s>>>(part, gamma, beta, coef, P, count, eps);
  profile_mark_begin(s);
  convt3d_apply_kernel<CIN><<<grid, block, 0, s>>>(x, w, b, coef, out, D, H, W);
  profile_mark_end(s);
}
// Tensor-core path (Cin <= 4): partials [N][4][P][kCtTcEpiWarps] float2 +
// coefficients.
struct CtTcWs {
  size_t part, coef, total;
  int P;  // tiles per sample
};

CtTcWs ct_tc_ws(int64_t N, int64_t D, int64_t H, int64_t W) {
  CtTcWs c{};
  c.P = int(D * ((H * W + 127) / 128));
  c.part = 0;
  c.coef = align_up(size_t(N) * kCT_G * c.P * kCtTcEpiWarps * sizeof(float2), 256);
  c.total = c.coef + align_up(size_t(N) * kCT_COUT * sizeof(float4), 256);
  return c;
}

template <int CIN>
gf_status launch_ct_tc_passes(const CtTcParams& prm, const float* gamma, const float* beta, float4* coef, int P,
                              int grid, float eps, cudaStream_t s) {
  if (cudaFuncSetAttribute(convt3d_tc_kernel<1, CIN>, cudaFuncAttributeMaxDynamicSharedMemorySize, kCtTcSmem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(convt3d_tc_kernel<2, CIN>, cudaFuncAttributeMaxDynamicSharedMemorySize, kCtTcSmem) !=
          cudaSuccess)
    return GF_ERR_CUDA;
  uint32_t* status = device_status_word();
  convt3d_tc_kernel<1, CIN><<<grid, kCtTcThreads, kCtTcSmem, s>>>(prm, status);
  const double count =
      double(kCT_COUT / kCT_G) * double(2 * prm.D - 1) * double(2 * prm.H - 1) * double(2 * prm.W - 1);
  convt3d_finalize_f2_kernel<<<dim3(unsigned(prm.N), kCT_G), 256, 0, s>>>(prm.part, gamma, beta, coef,
                                                                           P * kCtTcEpiWarps, count, eps);
  profile_mark_begin(s);
  convt3d_tc_kernel<2, CIN><<<grid, kCtTcThreads, kCtTcSmem, s>>>(prm, status);
  profile_mark_end(s);
  return cuda_status(cudaGetLastError());
}

// Single-kernel path: per-sample counters of finished tiles (zeroed by a
// memset before each launch) and per-tile slots of 8 partial sums.
struct CfWs {
  size_t done, part, total;
};

CfWs cf_ws(int64_t N, int64_t D, int64_t H, int64_t W) {
  const int64_t tiles = N * D * ((H * W + 127) / 128);
  CfWs c{};
  c.done = 0;
  c.part = align_up(size_t(N) * sizeof(uint32_t), 256);
  c.total = c.part + align_up(size_t(tiles) * 8 * sizeof(float), 256);
  return c;
}

template <int CIN>
gf_status launch_ct_fused(const CfParams& prm, int grid, cudaStream_t s) {
  if (cudaFuncSetAttribute(convt3d_fused_kernel<CIN>, cudaFuncAttributeMaxDynamicSharedMemorySize, kCfSmem) !=
      cudaSuccess)
    return GF_ERR_CUDA;
  uint32_t* status = device_status_word();
  CfParams p = prm;
  void* args[] = {&p, &status};
  profile_mark_begin(s);
  const cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(&convt3d_fused_kernel<CIN>),
                                                    dim3(unsigned(grid)), dim3(kCfThreads), args, kCfSmem, s);
  profile_mark_end(s);
  return cuda_status(e);
}

// The single-kernel path needs every CTA resident (one per SM), a sample of at
// most grid + 1 tiles (see convt3d_fused.cuh) and 16 channel volumes of a
// sample within 32-bit element offsets.
template <int CIN>
bool ct_fused_fits(int P, int grid, int device, uint64_t plane) {
  if (16 * plane >= (uint64_t(1) << 32)) return false;
  int coop = 0, blocks = 0;
  if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, device) != cudaSuccess || !coop) return false;
  if (cudaFuncSetAttribute(convt3d_fused_kernel<CIN>, cudaFuncAttributeMaxDynamicSharedMemorySize, kCfSmem) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, convt3d_fused_kernel<CIN>, kCfThreads, kCfSmem) !=
          cudaSuccess)
    return false;
  return blocks >= 1 && P <= grid + 1;
}

template <int CIN>
gf_status launch_ct_tensor_core(const float* x, const float* w, const float* b, const float* gamma,
                                const float* beta, float* out, int64_t N, int64_t D, int64_t H, int64_t W, float eps,
                                void* ws, const DeviceInfo& dev, cudaStream_t s) {
  const int bpp = int((H * W + 127) / 128), P = int(D) * bpp, num_tiles = int(N) * P;
  const int grid = num_tiles < dev.sm_count ? num_tiles : dev.sm_count;
  const uint64_t plane = uint64_t(2 * D - 1) * uint64_t(2 * H - 1) * uint64_t(2 * W - 1);
  if (ct_fused_fits<CIN>(P, grid, dev.device, plane)) {
    const CfWs cw = cf_ws(N, D, H, W);
    uint8_t* base = static_cast<uint8_t*>(ws);
    if (cudaMemsetAsync(base + cw.done, 0, cw.part - cw.done, s) != cudaSuccess) return GF_ERR_CUDA;
    CfParams p{};
    p.x = x;
    p.w = w;
    p.bias = b;
    p.gamma = gamma;
    p.beta = beta;
    p.out = out;
    p.part = reinterpret_cast<float*>(base + cw.part);
    p.done = reinterpret_cast<uint32_t*>(base + cw.done);
    p.N = int(N);
    p.D = int(D);
    p.H = int(H);
    p.W = int(W);
    p.bpp = bpp;
    p.num_tiles = num_tiles;
    p.rounds = (num_tiles + grid - 1) / grid;
    p.div_dp = make_fastdiv(uint32_t(P));
    p.div_bpp = make_fastdiv(uint32_t(bpp));
    p.div_w = make_fastdiv(uint32_t(W));
    p.inv_count = 1.0 / (double(kCT_COUT / kCT_G) * double(2 * D - 1) * double(2 * H - 1) * double(2 * W - 1));
    // the kernel's statistics are of s' = s log2 e (see convt3d_fused.cuh)
    p.eps = float(double(eps) * double(kLog2e) * double(kLog2e));
    p.plane = uint32_t(plane);
    p.OHW = int((2 * H - 1) * (2 * W - 1));
    p.OW = int(2 * W - 1);
    return launch_ct_fused<CIN>(p, grid, s);
  }
  const CtTcWs wl = ct_tc_ws(N, D, H, W);
  CtTcParams prm{};
  prm.x = x;
  prm.w = w;
  prm.bias = b;
  prm.part = reinterpret_cast<float2*>(static_cast<uint8_t*>(ws) + wl.part);
  float4* coef = reinterpret_cast<float4*>(static_cast<uint8_t*>(ws) + wl.coef);
  prm.coef = coef;
  prm.out = out;
  prm.N = int(N);
  prm.Cin = CIN;
  prm.D = int(D);
  prm.H = int(H);
  prm.W = int(W);
  prm.bpp = int((H * W + 127) / 128);
  prm.num_tiles = int(N * D * prm.bpp);
  prm.div_dp = make_fastdiv(uint32_t(D * prm.bpp));
  prm.div_bpp = make_fastdiv(uint32_t(prm.bpp));
  prm.div_w = make_fastdiv(uint32_t(W));
  return launch_ct_tc_passes<CIN>(prm, gamma, beta, coef, wl.P, grid, eps, s);
}

gf_status launch_ct_tc(const float* x, const float* w, const float* b, const float* gamma, const float* beta,
                       float* out, int64_t N, int64_t Cin, int64_t D, int64_t H, int64_t W, float eps, void* ws,
                       const DeviceInfo& dev, cudaStream_t s) {
  switch (Cin) {
    case 1: return launch_ct_tensor_core<1>(x, w, b, gamma, beta, out, N, D, H, W, eps, ws, dev, s);
    case 2: return launch_ct_tensor_core<2>(x, w, b, gamma, beta, out, N, D, H, W, eps, ws, dev, s);
    case 3: return launch_ct_tensor_core<3>(x, w, b, gamma, beta, out, N, D, H, W, eps, ws, dev, s);
    default: return launch_ct_tensor_core<4>(x, w, b, gamma, beta, out, N, D, H, W, eps, ws, dev, s);
  }
}
}  // namespace

// Fixed scratch for gf_convt3d_swish_gn_hswish_noalloc: the per-block GroupNorm
// partial sums and the per-channel affine coefficients live here instead of in
// a caller-provided workspace.  The array exists once per device that loads
// this library and is shared by every call of that entry point.
constexpr size_t kCtNoAllocScratchBytes = size_t(4) << 20;
static __device__ __align__(256) unsigned char g_ct_noalloc_scratch[kCtNoAllocScratchBytes];

namespace {
// An empty batch (N = 0): the arguments other than the batch are checked as
// for a batch of one (x and out may be NULL), then nothing is launched.
gf_status ct_empty_batch(const float* x, const float* w, const float* b, const float* gamma, const float* beta,
                         const float* out, int64_t Cin, int64_t Cout, int64_t D, int64_t H, int64_t W, int32_t k,
                         int32_t stride, int32_t pad, int32_t groups, float eps) {
  if (!w || !gamma || !beta) return GF_ERR_NULL;
  CtGenShape gen;
  if (check_ct_shape(1, Cin, Cout, D, H, W, k, stride, pad, groups) != GF_OK &&
      ct_general_shape(1, Cin, Cout, D, H, W, k, stride, pad, groups, &gen) != GF_OK)
    return GF_ERR_SHAPE;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return GF_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(w) || !aligned16(gamma) || !aligned16(beta) || !aligned16(out) ||
      (b && !aligned16(b)))
    return GF_ERR_ALIGN;
  return GF_OK;
}

std::mutex g_ct_scratch_mu;
void* g_ct_scratch_addr[64];
unsigned long long g_ct_scratch_ctx[64];

// Device address of g_ct_noalloc_scratch on the current device, looked up once
// per device and context.  In host code the array's name is only a host-side
// stand-in, so the kernels must be given this address instead.  The cached
// address is tied to the context it was looked up in (its unique id): after
// the context is destroyed and recreated (cudaDeviceReset) the module is
// loaded afresh and the address is looked up again.
gf_status ct_scratch_address(int device, void** addr) {
  if (device < 0 || device >= 64) return GF_ERR_CUDA;
  unsigned long long ctx = 0;
  if (current_context_id(&ctx) != GF_OK) return GF_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_ct_scratch_mu);
  if (!g_ct_scratch_addr[device] || g_ct_scratch_ctx[device] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ct_noalloc_scratch) != cudaSuccess || !p) return GF_ERR_CUDA;
    g_ct_scratch_addr[device] = p;
    g_ct_scratch_ctx[device] = ctx;
  }
  *addr = g_ct_scratch_addr[device];
  return GF_OK;
}

// Scratch bytes the no-workspace call needs for a shape (0: shape rejected):
// the CUDA-core two-pass kernels' partials and coefficients for the pages'
// configuration, the general kernels' workspace for every other shape.
size_t ct_noalloc_scratch_bytes(int64_t N, int64_t Cin, int64_t Cout, int64_t D, int64_t H, int64_t W, int32_t k,
                                int32_t stride, int32_t pad, int32_t groups) {
  if (N == 0) return 0;
  if (check_ct_shape(N, Cin, Cout, D, H, W, k, stride, pad, groups) == GF_OK) return ct_ws(N, D, H, W).total;
  CtGenShape g;
  return ct_general_shape(N, Cin, Cout, D, H, W, k, stride, pad, groups, &g) == GF_OK ? g.total : 0;
}
}  // namespace
}  // namespace gf

using namespace gf;

extern "C" {

size_t gf_convt3d_swish_gn_hswish_workspace_size(int64_t N, int64_t Cin, int64_t Cout, int64_t D, int64_t H,
                                                 int64_t W, int32_t k, int32_t stride, int32_t pad, int32_t groups) {
  if (N == 0) return 0;  // an empty batch launches nothing
  if (check_ct_shape(N, Cin, Cout, D, H, W, k, stride, pad, groups) != GF_OK) {
    // any other kernel size, stride, padding, channel counts or groups
    CtGenShape g;
    return ct_general_shape(N, Cin, Cout, D, H, W, k, stride, pad, groups, &g) == GF_OK ? g.total : 0;
  }
  if (Cin > 4) return ct_ws(N, D, H, W).total;
  // the single-kernel or the two-pass tensor-core path, chosen per device
  const size_t a = ct_tc_ws(N, D, H, W).total, c = cf_ws(N, D, H, W).total;
  return a > c ? a : c;
}

gf_status gf_convt3d_swish_gn_hswish(const float* x, const float* w, const float* b, const float* gamma,
                                     const float* beta, float* out, int64_t N, int64_t Cin, int64_t Cout, int64_t D,
                                     int64_t H, int64_t W, int32_t k, int32_t stride, int32_t pad, int32_t groups,
                                     float eps, void* workspace, size_t workspace_bytes, void* stream) {
  if (N == 0) return ct_empty_batch(x, w, b, gamma, beta, out, Cin, Cout, D, H, W, k, stride, pad, groups, eps);
  if (!x || !w || !gamma || !beta || !out) return GF_ERR_NULL;
  CtGenShape gen;
  const bool fast = check_ct_shape(N, Cin, Cout, D, H, W, k, stride, pad, groups) == GF_OK;
  gf_status st = fast ? GF_OK : ct_general_shape(N, Cin, Cout, D, H, W, k, stride, pad, groups, &gen);
  if (st != GF_OK) return st;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return GF_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(w) || !aligned16(gamma) || !aligned16(beta) || !aligned16(out) ||
      (b && !aligned16(b)) || !aligned16(workspace))
    return GF_ERR_ALIGN;
  const size_t need = gf_convt3d_swish_gn_hswish_workspace_size(N, Cin, Cout, D, H, W, k, stride, pad, groups);
  if (!fast) {
    if (!workspace) return GF_ERR_NULL;
    if (workspace_bytes < need) return GF_ERR_WORKSPACE;
    const Span gins[] = {{x, size_t(N) * Cin * D * H * W * 4},
                         {w, size_t(Cin) * Cout * k * k * k * 4},
                         {b, size_t(Cout) * 4},
                         {gamma, size_t(Cout) * 4},
                         {beta, size_t(Cout) * 4},
                         {workspace, need}};
    st = check_no_alias(Span{out, size_t(N) * Cout * gen.OD * gen.OH * gen.OW * 4}, gins, 6);
    if (st != GF_OK) return st;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != GF_OK) return st;
    return launch_ct_general(gen, x, w, b, gamma, beta, out, eps, workspace, static_cast<cudaStream_t>(stream));
  }
  if (!workspace) return GF_ERR_NULL;
  if (workspace_bytes < need) return GF_ERR_WORKSPACE;
  const size_t outb = size_t(N) * Cout * (2 * D - 1) * (2 * H - 1) * (2 * W - 1) * 4;
  const Span ins[] = {{x, size_t(N) * Cin * D * H * W * 4},
                      {w, size_t(Cin) * Cout * 27 * 4},
                      {b, size_t(Cout) * 4},
                      {gamma, size_t(Cout) * 4},
                      {beta, size_t(Cout) * 4},
                      {workspace, need}};
  st = check_no_alias(Span{out, outb}, ins, 6);
  if (st != GF_OK) return st;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != GF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Cin <= 4: the contraction runs on the tensor cores (K = 8 Cin <= 32)
  if (Cin <= 4) return launch_ct_tc(x, w, b, gamma, beta, out, N, Cin, D, H, W, eps, workspace, dev, s);
  const CtWs wl = ct_ws(N, D, H, W);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  double* part = reinterpret_cast<double*>(ws + wl.part);
  float2* coef = reinterpret_cast<float2*>(ws + wl.coef);
  const int n = int(N), d = int(D), h = int(H), ww = int(W);
  switch (Cin) {
#define GF_CT_CASE(c) \
  case c: launch_ct<c>(x, w, b, part, gamma, beta, coef, out, n, d, h, ww, wl.P, eps, s); break;
    GF_CT_CASE(1) GF_CT_CASE(2) GF_CT_CASE(3) GF_CT_CASE(4) GF_CT_CASE(5) GF_CT_CASE(6) GF_CT_CASE(7) GF_CT_CASE(8)
#undef GF_CT_CASE
    default: return GF_ERR_SHAPE;
  }
  return cuda_status(cudaGetLastError());
}

size_t gf_convt3d_noalloc_scratch_limit(void) { return kCtNoAllocScratchBytes; }

size_t gf_convt3d_swish_gn_hswish_noalloc_scratch_size(int64_t N, int64_t Cin, int64_t Cout, int64_t D, int64_t H,
                                                       int64_t W, int32_t k, int32_t stride, int32_t pad,
                                                       int32_t groups) {
  return ct_noalloc_scratch_bytes(N, Cin, Cout, D, H, W, k, stride, pad, groups);
}

gf_status gf_convt3d_swish_gn_hswish_noalloc(const float* x, const float* w, const float* b, const float* gamma,
                                             const float* beta, float* out, int64_t N, int64_t Cin, int64_t Cout,
                                             int64_t D, int64_t H, int64_t W, int32_t k, int32_t stride, int32_t pad,
                                             int32_t groups, float eps, void* stream) {
  if (N == 0) return ct_empty_batch(x, w, b, gamma, beta, out, Cin, Cout, D, H, W, k, stride, pad, groups, eps);
  if (!x || !w || !gamma || !beta || !out) return GF_ERR_NULL;
  CtGenShape gen;
  const bool fast = check_ct_shape(N, Cin, Cout, D, H, W, k, stride, pad, groups) == GF_OK;
  gf_status st = fast ? GF_OK : ct_general_shape(N, Cin, Cout, D, H, W, k, stride, pad, groups, &gen);
  if (st != GF_OK) return st;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return GF_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(w) || !aligned16(gamma) || !aligned16(beta) || !aligned16(out) ||
      (b && !aligned16(b)))
    return GF_ERR_ALIGN;
  if (ct_noalloc_scratch_bytes(N, Cin, Cout, D, H, W, k, stride, pad, groups) > kCtNoAllocScratchBytes)
    return GF_ERR_WORKSPACE;  // beyond the fixed scratch
  if (!fast) {  // the general kernels, their workspace in the fixed scratch
    const Span gins[] = {{x, size_t(N) * Cin * D * H * W * 4},
                         {w, size_t(Cin) * Cout * k * k * k * 4},
                         {b, size_t(Cout) * 4},
                         {gamma, size_t(Cout) * 4},
                         {beta, size_t(Cout) * 4}};
    st = check_no_alias(Span{out, size_t(N) * Cout * gen.OD * gen.OH * gen.OW * 4}, gins, 5);
    if (st != GF_OK) return st;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != GF_OK) return st;
    void* scratch = nullptr;
    if ((st = ct_scratch_address(dev.device, &scratch)) != GF_OK) return st;
    return launch_ct_general(gen, x, w, b, gamma, beta, out, eps, scratch, static_cast<cudaStream_t>(stream));
  }
  const CtWs wl = ct_ws(N, D, H, W);
  const size_t outb = size_t(N) * Cout * (2 * D - 1) * (2 * H - 1) * (2 * W - 1) * 4;
  const Span ins[] = {{x, size_t(N) * Cin * D * H * W * 4},
                      {w, size_t(Cin) * Cout * 27 * 4},
                      {b, size_t(Cout) * 4},
                      {gamma, size_t(Cout) * 4},
                      {beta, size_t(Cout) * 4}};
  st = check_no_alias(Span{out, outb}, ins, 5);
  if (st != GF_OK) return st;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != GF_OK) return st;
  void* scratch = nullptr;
  if ((st = ct_scratch_address(dev.device, &scratch)) != GF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(scratch);
  double* part = reinterpret_cast<double*>(ws + wl.part);
  float2* coef = reinterpret_cast<float2*>(ws + wl.coef);
  const int n = int(N), d = int(D), h = int(H), ww = int(W);
  switch (Cin) {
#define GF_CT_CASE(c) \
  case c: launch_ct<c>(x, w, b, part, gamma, beta, coef, out, n, d, h, ww, wl.P, eps, s); break;
    GF_CT_CASE(1) GF_CT_CASE(2) GF_CT_CASE(3) GF_CT_CASE(4) GF_CT_CASE(5) GF_CT_CASE(6) GF_CT_CASE(7) GF_CT_CASE(8)
#undef GF_CT_CASE
    default: return GF_ERR_SHAPE;
  }
  return cuda_status(cudaGetLastError());
}

}  // extern "C"
