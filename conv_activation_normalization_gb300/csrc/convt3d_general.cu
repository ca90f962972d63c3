// ConvTranspose3d -> Swish -> GroupNorm -> HardSwish for any kernel size,
// stride, padding, channel counts and groups   (page Kimi-K2.6__l2_p60)
//
// Gather form of the transposed convolution: output o (per dimension)
// receives x[i] w[k] for every tap k with o = S i - Pd + k, i.e. the taps
// k = k0 + j S with k0 = (o + Pd) mod S, whose input i = (o + Pd - k) / S
// falls inside the input; those j form one contiguous range.
//   pass 1  one thread per output voxel and chunk of 8 channels: conv +
//           bias + Swish, per-thread fp64 (sum, sum of squares) per channel,
//           reduced per block and written per (sample, channel, block);
//   finalize per (sample, group): fp64 mean and biased variance over the
//           group's channels -> A = gamma rstd, B = beta - mean A per channel;
//   pass 2  recompute, HardSwish(A s + B), store (coalesced along the voxel).
// The weights are read through the read-only cache; this path serves the
// shapes the tensor-core kernels do not take, not the pages' workload.
#include <cmath>

#include "convt3d_general.h"
#include "host_common.h"

namespace gf {
namespace {

constexpr int kCgThreads = 256;
constexpr int kCgChunk = 8;  // output channels per sweep over the voxels

struct CgParams {
  const float* x;
  const float* w;
  const float* b;  // may be null
  const float* gamma;
  const float* beta;
  float* out;
  double* part;    // [N][Cout][P][2]
  float2* coef;    // [N][Cout]: (A, B)
  int Cin, Cout, G, D, H, W, K, S, Pd, OD, OH, OW, P;
  float eps;
};

// Taps of output index o along one dimension: k = k0 + j S and input
// i = itop - j for j0 <= j < j1.
struct Taps {
  int k0, itop, j0, j1;
};
__device__ __forceinline__ Taps taps_1d(int o, int I, int K, int S, int Pd) {
  Taps t;
  const int q = o + Pd;  // >= 0
  t.k0 = q % S;
  t.itop = (q - t.k0) / S;                     // input of tap k0
  t.j0 = t.itop >= I ? t.itop - I + 1 : 0;    // i = itop - j < I
  const int jk = (K - t.k0 + S - 1) / S;       // k0 + j S < K
  t.j1 = min(jk, t.itop + 1);                  // i >= 0
  return t;
}

// y of channels c0 .. c0 + 7 at output voxel (od, oh, ow) of sample n (bias
// included; channels past Cout are left at 0).
__device__ __forceinline__ void conv_voxel(const CgParams& p, int n, int c0, int od, int oh, int ow,
                                           float (&y)[kCgChunk]) {
#pragma unroll
  for (int j = 0; j < kCgChunk; ++j) y[j] = (p.b && c0 + j < p.Cout) ? __ldg(p.b + c0 + j) : 0.f;
  const Taps td = taps_1d(od, p.D, p.K, p.S, p.Pd), th = taps_1d(oh, p.H, p.K, p.S, p.Pd),
             tw = taps_1d(ow, p.W, p.K, p.S, p.Pd);
  const size_t HW = size_t(p.H) * p.W, DHW = HW * p.D, K3 = size_t(p.K) * p.K * p.K;
  const float* xn = p.x + size_t(n) * p.Cin * DHW;
  const int nch = min(kCgChunk, p.Cout - c0);
  for (int jd = td.j0; jd < td.j1; ++jd) {
    const int kd = td.k0 + jd * p.S, id = td.itop - jd;
    for (int jh = th.j0; jh < th.j1; ++jh) {
      const int kh = th.k0 + jh * p.S, ih = th.itop - jh;
      for (int jw = tw.j0; jw < tw.j1; ++jw) {
        const int kw = tw.k0 + jw * p.S, iw = tw.itop - jw;
        const size_t xo = (size_t(id) * p.H + ih) * p.W + iw;
        const size_t wo = (size_t(kd) * p.K + kh) * p.K + kw;
        for (int ci = 0; ci < p.Cin; ++ci) {
          const float xv = __ldg(xn + size_t(ci) * DHW + xo);
          // w[ci][co][kd][kh][kw]
          const float* wc = p.w + (size_t(ci) * p.Cout + c0) * K3 + wo;
#pragma unroll
          for (int j = 0; j < kCgChunk; ++j)
            if (j < nch) y[j] = fmaf(xv, __ldg(wc + size_t(j) * K3), y[j]);
        }
      }
    }
  }
}

__device__ __forceinline__ float swish(float y) { return y / (1.f + expf(-y)); }

// Block sum of one double per thread; the result is valid in thread 0.
__device__ __forceinline__ double block_sum(double v, double* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __syncthreads();  // red may still be read from the previous call
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double t = 0.0;
  if (threadIdx.x == 0)
    for (int i = 0; i < kCgThreads / 32; ++i) t += red[i];
  return t;
}

// grid (P, N): block b of sample n takes voxels b*256 + t, + P*256, ...
template <bool PASS2>
__global__ void __launch_bounds__(kCgThreads, 1) ct_general_kernel(const CgParams p) {
  __shared__ double red[kCgThreads / 32];
  const int n = blockIdx.y;
  const int ov = p.OD * p.OH * p.OW;  // < 2^30: no overflow below
  const int step = p.P * kCgThreads;
  for (int c0 = 0; c0 < p.Cout; c0 += kCgChunk) {
    double s1[kCgChunk], s2[kCgChunk];
    float2 ab[kCgChunk];
#pragma unroll
    for (int j = 0; j < kCgChunk; ++j) {
      s1[j] = s2[j] = 0.0;
      if constexpr (PASS2) ab[j] = c0 + j < p.Cout ? p.coef[size_t(n) * p.Cout + c0 + j] : make_float2(0.f, 0.f);
    }
    for (int v = blockIdx.x * kCgThreads + threadIdx.x; v < ov; v += step) {
      const int r = v / p.OW, ow = v - r * p.OW;
      const int od = r / p.OH, oh = r - od * p.OH;
      float y[kCgChunk];
      conv_voxel(p, n, c0, od, oh, ow, y);
#pragma unroll
      for (int j = 0; j < kCgChunk; ++j) {
        if (c0 + j >= p.Cout) break;
        const float sv = swish(y[j]);
        if constexpr (PASS2) {
          const float h = fmaf(ab[j].x, sv, ab[j].y);
          __stcs(p.out + (size_t(n) * p.Cout + c0 + j) * size_t(ov) + size_t(v),
                 h * fminf(fmaxf(h + 3.f, 0.f), 6.f) * (1.f / 6.f));
        } else {
          s1[j] += double(sv);
          s2[j] += double(sv) * double(sv);
        }
      }
    }
    if constexpr (!PASS2) {
#pragma unroll
      for (int j = 0; j < kCgChunk; ++j) {
        if (c0 + j >= p.Cout) break;  // uniform across the block
        const double a = block_sum(s1[j], red), q = block_sum(s2[j], red);
        if (threadIdx.x == 0) {
          double* d = p.part + ((size_t(n) * p.Cout + c0 + j) * p.P + blockIdx.x) * 2;
          d[0] = a;
          d[1] = q;
        }
      }
    }
  }
}

// grid N: per group, the fp64 totals over its channels and blocks, then the
// per-channel affine.
__global__ void __launch_bounds__(kCgThreads) ct_general_finalize_kernel(const CgParams p) {
  __shared__ double red[kCgThreads / 32];
  const int n = blockIdx.x, cg = p.Cout / p.G;
  const double count = double(cg) * p.OD * p.OH * p.OW;
  for (int g = 0; g < p.G; ++g) {
    double a = 0.0, q = 0.0;
    const double* base = p.part + size_t(n) * p.Cout * p.P * 2 + size_t(g) * cg * p.P * 2;
    for (int i = threadIdx.x; i < cg * p.P; i += kCgThreads) {
      a += base[2 * size_t(i)];
      q += base[2 * size_t(i) + 1];
    }
    a = block_sum(a, red);
    q = block_sum(q, red);
    __shared__ double mv[2];
    if (threadIdx.x == 0) {
      const double mean = a / count;
      mv[0] = mean;
      mv[1] = fmax(q / count - mean * mean, 0.0);
    }
    __syncthreads();
    for (int c = threadIdx.x; c < cg; c += kCgThreads) {
      const int co = g * cg + c;
      const double A = double(p.gamma[co]) / sqrt(mv[1] + double(p.eps));
      p.coef[size_t(n) * p.Cout + co] = make_float2(float(A), float(double(p.beta[co]) - mv[0] * A));
    }
    __syncthreads();  // mv is rewritten for the next group
  }
}

}  // namespace

gf_status ct_general_shape(int64_t N, int64_t Cin, int64_t Cout, int64_t D, int64_t H, int64_t W, int32_t k,
                           int32_t stride, int32_t pad, int32_t groups, CtGenShape* s) {
  if (k < 1 || k > 8 || stride < 1 || stride > 8 || pad < 0 || pad > 64) return GF_ERR_SHAPE;
  if (N < 1 || N > 65535 || Cin < 1 || Cin > 1024 || Cout < 1 || Cout > 1024) return GF_ERR_SHAPE;
  if (groups < 1 || Cout % groups != 0) return GF_ERR_SHAPE;
  if (D < 1 || H < 1 || W < 1 || D > (1 << 20) || H > (1 << 20) || W > (1 << 20)) return GF_ERR_SHAPE;
  const auto osz = [&](int64_t I) { return (I - 1) * stride - 2 * int64_t(pad) + k; };
  const int64_t OD = osz(D), OH = osz(H), OW = osz(W);
  if (OD < 1 || OH < 1 || OW < 1) return GF_ERR_SHAPE;
  if (OD * OH * OW >= (int64_t(1) << 30) || Cin * D * H * W >= (int64_t(1) << 31)) return GF_ERR_SHAPE;
  s->N = N, s->Cin = Cin, s->Cout = Cout, s->D = D, s->H = H, s->W = W;
  s->K = k, s->S = stride, s->Pd = pad, s->G = groups;
  s->OD = OD, s->OH = OH, s->OW = OW;
  // blocks per sample: enough for the voxels, at most about 4096 blocks in all
  const int64_t need = (OD * OH * OW + kCgThreads - 1) / kCgThreads;
  const int64_t cap = N >= 4096 ? 1 : 4096 / N;
  s->P = int(need < cap ? need : cap);
  s->part = 0;
  s->coef = align_up(size_t(N) * Cout * s->P * 2 * sizeof(double), 256);
  s->total = s->coef + align_up(size_t(N) * Cout * sizeof(float2), 256);
  return GF_OK;
}

gf_status launch_ct_general(const CtGenShape& s, const float* x, const float* w, const float* b, const float* gamma,
                            const float* beta, float* out, float eps, void* workspace, cudaStream_t stream) {
  CgParams p;
  p.x = x, p.w = w, p.b = b, p.gamma = gamma, p.beta = beta, p.out = out;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.part = reinterpret_cast<double*>(ws + s.part);
  p.coef = reinterpret_cast<float2*>(ws + s.coef);
  p.Cin = int(s.Cin), p.Cout = int(s.Cout), p.G = s.G, p.D = int(s.D), p.H = int(s.H), p.W = int(s.W);
  p.K = s.K, p.S = s.S, p.Pd = s.Pd, p.OD = int(s.OD), p.OH = int(s.OH), p.OW = int(s.OW), p.P = s.P;
  p.eps = eps;
  const dim3 grid(unsigned(s.P), unsigned(s.N));
  ct_general_kernel<false><<<grid, kCgThreads, 0, stream>>>(p);
  ct_general_finalize_kernel<<<unsigned(s.N), kCgThreads, 0, stream>>>(p);
  profile_mark_begin(stream);
  ct_general_kernel<true><<<grid, kCgThreads, 0, stream>>>(p);
  profile_mark_end(stream);
  return cuda_status(cudaGetLastError());
}

}  // namespace gf
