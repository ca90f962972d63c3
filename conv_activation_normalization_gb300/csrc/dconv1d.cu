// LayerNorm([C, L]) -> GELU -> dilated Conv1d -> +x   (page Kimi-K2.6__l2_p5)
//
//   1. ln_partial:   per (sample, chunk of 8192 elements) the shifted sums
//                    S1, S2 about one shift per sample: fp32 per thread and
//                    warp, fp64 across warps;
//   2. ln_finalize:  per sample, fp64 sum of the partials -> (mean, rstd);
//   3. ln_apply:     a = GELU((x - mean) * rstd * gamma + beta), transposed to
//                    [B][L][C] through shared memory and split into TF32 hi/lo
//                    planes, the K-major A operand of the implicit GEMM;
//   4. weight split: W[co][ci][t] -> planes[co][t * C + ci];
//   5. the tcgen05 3xTF32 implicit GEMM (ConvSrc): the three dilated taps are
//      TMA boxes of the same activation planes shifted by dilation along L,
//      with the TMA unit's zero fill supplying the padding; its epilogue adds
//      the conv bias and the residual x and stores out[b][co][j] (32
//      consecutive j per warp, so every store is a full 128-byte line).
//
// With GF_FLAG_FUSED_PRODUCER (3xTF32 mode, taps spanning at most 92
// positions) steps 3-5 are one kernel instead (LnConvSrc): converter warps
// inside the GEMM apply LayerNorm and GELU to raw x while they build each
// stage's A operand, so the activation planes are never written and the
// workspace shrinks from 8 B per activation to the statistics and weight
// planes; steps 1, 2 and a weight split remain.  It is the slower path on
// the benchmark workload (0.46 against 0.32 ms per call): the window of
// activations it computes per tile and channel block cannot be
// double-buffered within the shared memory the two 96 KB stages leave, so
// its LayerNorm/GELU work does not overlap the MMAs, and the planes path
// stays the default.
#include <cmath>
#include <type_traits>

#include "gemm_tc.cuh"
#include "host_common.h"
#include "kernels_common.cuh"

namespace gf {

constexpr int kLnChunk = 8192;  // elements per ln_partial block (256 threads x 32)
// In the 3xTF32 mode the GEMM computes the activations' lo plane in the SM
// (gemm_tc_kernel, kLoInSm) while the weight planes are still arriving, so
// the LayerNorm pass writes only the raw fp32 plane (step 0.2986 -> 0.2858
// ms on x[32,256,4096]; the GEMM's time is unchanged).  The weights keep
// both planes: converting them too made the GEMM slower (0.330 ms steps).
constexpr int kLoConv = 1;

// The statistics of a sample are taken as shifted sums S1 = sum (x - c) and
// S2 = sum (x - c)^2 about one shift c per sample (the mean of the sample's
// first 32 values, which every block computes identically).  With a common
// shift the sums are additive, so they are reduced in fp32 within a thread
// and a warp and in fp64 across warps and blocks; c near the data keeps
// var = S2/n - (S1/n)^2 well conditioned.
__device__ __forceinline__ float sample_shift(const float* __restrict__ xs, int64_t n_per_sample) {
  const int lane = threadIdx.x & 31;
  float v = lane < n_per_sample ? __ldg(xs + lane) : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v / float(n_per_sample < 32 ? n_per_sample : 32);
}

// grid (chunks, B), 256 threads.  n_per_sample = C * L; VEC: float4 loads
// (n_per_sample a multiple of 4, so every sample starts 16-byte aligned),
// else scalar.  part[b][chunk] = (S1, S2) of the chunk's elements, in fp64.
template <bool VEC>
__global__ void __launch_bounds__(256) ln_partial_kernel(const float* __restrict__ x, double2* __restrict__ part,
                                                         int64_t n_per_sample, int chunks) {
  __shared__ double2 red[8];
  const int b = blockIdx.y;
  const float* xs = x + size_t(b) * size_t(n_per_sample);
  const int64_t begin = int64_t(blockIdx.x) * kLnChunk;
  const int64_t end = begin + kLnChunk < n_per_sample ? begin + kLnChunk : n_per_sample;
  float s1 = 0.f, s2 = 0.f;
  if constexpr (VEC) {
    // all of the thread's loads (kLnChunk / 1024 float4) are issued before
    // any arithmetic, so that they and the shift's own load overlap
    constexpr int kPer = kLnChunk / (4 * 256);
    float4 v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int64_t i = begin + 4 * (threadIdx.x + int64_t(u) * blockDim.x);
      v[u] = i < end ? __ldcs(reinterpret_cast<const float4*>(xs + i)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float shift = sample_shift(xs, n_per_sample);
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int64_t i = begin + 4 * (threadIdx.x + int64_t(u) * blockDim.x);
      if (i < end) {
        const float d0 = v[u].x - shift, d1 = v[u].y - shift, d2 = v[u].z - shift, d3 = v[u].w - shift;
        s1 += (d0 + d1) + (d2 + d3);
        s2 += fmaf(d0, d0, d1 * d1) + fmaf(d2, d2, d3 * d3);
      }
    }
  } else {
    const float shift = sample_shift(xs, n_per_sample);
    for (int64_t i = begin + threadIdx.x; i < end; i += blockDim.x) {
      const float d = __ldcs(xs + i) - shift;
      s1 += d;
      s2 = fmaf(d, d, s2);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s1 += __shfl_xor_sync(0xffffffffu, s1, o);
    s2 += __shfl_xor_sync(0xffffffffu, s2, o);
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = make_double2(s1, s2);
  __syncthreads();
  if (threadIdx.x == 0) {
    double a = 0.0, q = 0.0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      a += red[w].x;
      q += red[w].y;
    }
    part[size_t(b) * chunks + blockIdx.x] = make_double2(a, q);
  }
}

// One block of 256 threads: sum sample b's partials -> (mean, rstd).
__device__ __forceinline__ void ln_finalize_block(const float* __restrict__ x, const double2* __restrict__ part,
                                                  float2* __restrict__ stats, int64_t n_per_sample, int chunks,
                                                  float eps, int b) {
  __shared__ double2 red[8];
  double a = 0.0, q = 0.0;
  for (int i = threadIdx.x; i < chunks; i += blockDim.x) {
    const double2 p = part[size_t(b) * chunks + i];
    a += p.x;
    q += p.y;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    q += __shfl_xor_sync(0xffffffffu, q, o);
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = make_double2(a, q);
  const float shift = sample_shift(x + size_t(b) * size_t(n_per_sample), n_per_sample);
  __syncthreads();
  if (threadIdx.x == 0) {
    double A = 0.0, Q = 0.0;
    for (int w = 0; w < 8; ++w) {
      A += red[w].x;
      Q += red[w].y;
    }
    const double n = double(n_per_sample);
    const double m = A / n;
    const double var = fmax(Q / n - m * m, 0.0);
    stats[b] = make_float2(float(double(shift) + m), float(1.0 / sqrt(var + double(eps))));
  }
}

// Writes the GEMM operand planes of one activation / weight value v at
// element offset o: 3xTF32 -> fp32 (v, v - tf32_hi(v)) (the tensor core reads
// v itself as hi); BF16 -> bf16(v); 3xBF16 -> bf16 hi and bf16(v - hi).
template <int MODE>
__device__ __forceinline__ void store_planes(void* planes, size_t plane_elems, size_t o, float v) {
  if constexpr (MODE == GF_MODE_FP32_3XTF32) {
    float* p = static_cast<float*>(planes);
    p[o] = v;
    p[plane_elems + o] = v - tf32_hi(v);
  } else {
    __nv_bfloat16* p = static_cast<__nv_bfloat16*>(planes);
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    p[o] = h;
    if constexpr (MODE == GF_MODE_FP32_3XBF16) p[plane_elems + o] = __float2bfloat16_rn(v - __bfloat162float(h));
  }
}

// The operand planes of 4 consecutive channels (element offset o, a
// multiple of 4): one 16-byte store per fp32 plane, 8 bytes per bf16 plane.
template <int MODE>
__device__ __forceinline__ void store_planes4(void* planes, size_t plane_elems, size_t o, float4 v) {
  if constexpr (MODE == GF_MODE_FP32_3XTF32) {
    float* p = static_cast<float*>(planes);
    __stcs(reinterpret_cast<float4*>(p + o), v);
    if constexpr (!(kLoConv & 1))  // (else the GEMM computes the lo plane itself)
      __stcs(reinterpret_cast<float4*>(p + plane_elems + o),
             make_float4(v.x - tf32_hi(v.x), v.y - tf32_hi(v.y), v.z - tf32_hi(v.z), v.w - tf32_hi(v.w)));
  } else {
    __nv_bfloat16* p = static_cast<__nv_bfloat16*>(planes);
    Bf16x4 h, l;
    bf16_split4(v, h, l);
    *reinterpret_cast<Bf16x4*>(p + o) = h;
    if constexpr (MODE == GF_MODE_FP32_3XBF16) *reinterpret_cast<Bf16x4*>(p + plane_elems + o) = l;
  }
}

// grid (ceil(L/128), Cp/32, B), 256 threads: GELU(LayerNorm(x)) for a tile
// of 32 channels x 128 positions, read as float4 along L (x, gamma, beta),
// transposed through shared memory and written 4 channels at a time to the
// [B][L][Cp] operand planes; channels C .. Cp - 1 (the padding to a whole
// number of k-blocks) are written as zeros.  VEC: float4 loads (L a multiple
// of 4, rows 16-byte aligned), else scalar.  TANH: GELU's tanh approximation
// instead of the erf form.
template <int MODE, bool TANH, bool VEC>
__global__ void __launch_bounds__(256) ln_apply_gelu_split_kernel(const float* __restrict__ x,
                                                                  const float* __restrict__ gamma,
                                                                  const float* __restrict__ beta,
                                                                  const float2* __restrict__ stats, void* planes,
                                                                  int C, int Cp, int L, int B) {
  __shared__ __align__(16) float tile[32][132];  // [channel][position]; 16-byte rows, 4-way reads
  const int l0 = blockIdx.x * 128, c0 = blockIdx.y * 32, b = blockIdx.z;
  const float2 st = stats[b];
  const int t = threadIdx.x;
  const float* xb = x + size_t(b) * C * L;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int item = t + 256 * i, cc = item >> 5, q = item & 31;  // a warp: one channel, 128 positions
    const int l = l0 + 4 * q;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (l < L && c0 + cc < C) {
      const size_t cl = size_t(c0 + cc) * L + l;
      float4 v, g, be;
      if constexpr (VEC) {
        v = __ldcs(reinterpret_cast<const float4*>(xb + cl));
        g = __ldg(reinterpret_cast<const float4*>(gamma + cl));
        be = __ldg(reinterpret_cast<const float4*>(beta + cl));
      } else {  // positions past L load as 0 and are not stored
        float e[3][4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const bool in = l + k < L;
          e[0][k] = in ? __ldcs(xb + cl + k) : 0.f;
          e[1][k] = in ? __ldg(gamma + cl + k) : 0.f;
          e[2][k] = in ? __ldg(beta + cl + k) : 0.f;
        }
        v = make_float4(e[0][0], e[0][1], e[0][2], e[0][3]);
        g = make_float4(e[1][0], e[1][1], e[1][2], e[1][3]);
        be = make_float4(e[2][0], e[2][1], e[2][2], e[2][3]);
      }
      const float4 h = make_float4(fmaf((v.x - st.x) * st.y, g.x, be.x), fmaf((v.y - st.x) * st.y, g.y, be.y),
                                   fmaf((v.z - st.x) * st.y, g.z, be.z), fmaf((v.w - st.x) * st.y, g.w, be.w));
      if constexpr (TANH)
        a = make_float4(gelu_tanh(h.x), gelu_tanh(h.y), gelu_tanh(h.z), gelu_tanh(h.w));
      else
        a = make_float4(gelu_erf(h.x), gelu_erf(h.y), gelu_erf(h.z), gelu_erf(h.w));
    }
    *reinterpret_cast<float4*>(&tile[cc][4 * q]) = a;
  }
  __syncthreads();
  const size_t plane = size_t(B) * L * Cp;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int item = t + 256 * i, pl = item >> 3, cq = item & 7;  // a warp: 4 positions x 32 channels
    const int l = l0 + pl;
    if (l < L)
      store_planes4<MODE>(planes, plane, (size_t(b) * L + l) * Cp + c0 + 4 * cq,
                          make_float4(tile[4 * cq][pl], tile[4 * cq + 1][pl], tile[4 * cq + 2][pl],
                                      tile[4 * cq + 3][pl]));
  }
}

// W[co][ci][t] -> planes[Cout][ksize * Cp] in the GEMM's k order: k-block
// kb = cb * ksize + t holds channels cb * BK .. + BK - 1 of tap t (BK = 32
// fp32 or 64 bf16 elements, one 128-byte row), zeros for the padding
// channels C .. Cp - 1.  Block `blk` of `nblk` (grid-stride over elements).
template <int MODE>
__device__ __forceinline__ void conv_weight_split_blocks(const float* __restrict__ w, void* planes, int Cout, int C,
                                                         int Cp, int ksize, int blk, int nblk) {
  constexpr int BK = MODE == GF_MODE_FP32_3XTF32 ? 32 : 64;
  const int64_t n = int64_t(Cout) * ksize * Cp;
  for (int64_t i = int64_t(blk) * blockDim.x + threadIdx.x; i < n; i += int64_t(nblk) * blockDim.x) {
    const int64_t co = i / (int64_t(ksize) * Cp);
    const int k = int(i - co * (int64_t(ksize) * Cp));
    const int kb = k / BK, c = k % BK;
    const int cb = kb / ksize, t = kb - cb * ksize;
    const int ci = cb * BK + c;
    store_planes<MODE>(planes, size_t(n), size_t(i), ci < C ? w[(co * C + ci) * ksize + t] : 0.f);
  }
}

// grid B + weight blocks, 256 threads: blocks b < B finalize sample b's
// LayerNorm statistics, the others split the conv weights into the GEMM's
// operand planes.  The two jobs are independent and each is too small to
// fill the GPU, so one launch runs them side by side.
template <int MODE>
__global__ void __launch_bounds__(256) ln_finalize_weights_kernel(const float* __restrict__ x,
                                                                  const double2* __restrict__ part,
                                                                  float2* __restrict__ stats, int64_t n_per_sample,
                                                                  int chunks, float eps, int B,
                                                                  const float* __restrict__ w, void* w_planes, int C,
                                                                  int Cp, int ksize) {
  if (int(blockIdx.x) < B)
    ln_finalize_block(x, part, stats, n_per_sample, chunks, eps, int(blockIdx.x));
  else
    conv_weight_split_blocks<MODE>(w, w_planes, C, C, Cp, ksize, int(blockIdx.x) - B, int(gridDim.x) - B);
}

// Operand source of the fused LayerNorm -> GELU -> dilated Conv1d GEMM (3xTF32
// mode): rows are output positions j of one sample, columns output channels,
// and the reduction runs over channel blocks cb of 32 (outer) and taps t
// (inner), k-block kb = cb * ksize + t; the weight planes are laid out in that
// order (conv_weight_split_blocks, as for the planes path).  Warp 0 loads
// only the weights (B); five converter warps build A.  Per tile and channel block they compute the
// activation a = GELU((x - mean) rstd gamma + beta) once for the window of
// positions l = j0 - pad + p, p < 128 + (ksize - 1) dil (zero outside
// [0, L): the conv's padding), into shared memory (128-byte rows of 32
// channels, 16-byte chunks swizzled by row; the window starts at the 4-aligned
// position at or before j0 - pad, `shift` rows earlier), then four of them
// copy, for each tap, window rows shift + t dil .. + 127 into the stage's A
// planes (hi = the value, which the tensor core truncates; lo = value - its
// TF32 part).  A window task is 4 positions x 4 channels: x, gamma and beta
// each read as 4 float4 (all 12 loads issued before any arithmetic), so that
// many loads are in flight per thread.
template <bool TANH>
struct LnConvSrc {
  static constexpr int kConverterWarps = 5;
  static constexpr int kArrivingWarps = 4;                      // the copying warps: one A row per thread
  static constexpr int kMaxWindow = 220;                        // positions: 128 + (ksize - 1) dil <= 220
  static constexpr int kScratchBytes = (kMaxWindow + 4) * 128;  // + the alignment shift
  const float* x;
  const float* gamma;
  const float* beta;
  const float2* stats;  // [B] (mean, rstd)
  int C, Cp, L, pad, dil, ksize;
  int num_jb, num_nb, num_kb, bn, bk, nsamples;
  int kb_chunk;
  int ncb;      // Cp / 32
  int wrows;    // 128 + (ksize - 1) dil
  __device__ __forceinline__ int num_tiles() const { return nsamples * num_jb * num_nb; }
  __device__ __forceinline__ Tile tile(int t) const {
    const int nb = t % num_nb;
    const int r = t / num_nb;
    const int jb = r % num_jb;
    const int b = r / num_jb;
    return Tile{b, jb * kBM, nb * bn, nb};
  }
  template <int PLANES>
  __device__ __forceinline__ void load(const OperandMaps& m, uint64_t* bar, const uint32_t*, const uint32_t* sb,
                                       const Tile& t, int kb) const {
#pragma unroll
    for (int p = 0; p < PLANES; ++p) tma_load_2d(sb[p], &m.b[p], bar, kb * bk, t.n0);
  }
  // byte offset of 16-byte chunk q of row r in a 128-byte-row swizzled tile
  __device__ __forceinline__ static uint32_t chunk_off(int r, int q) {
    return uint32_t(r) * 128u + ((uint32_t(q) ^ uint32_t(r & 7)) << 4);
  }
  __device__ __forceinline__ static float act(float h) { return TANH ? gelu_tanh(h) : gelu_erf(h); }

  // one window task: positions pos0 .. pos0 + 3 (window rows row0 .. row0 + 3)
  // x channels c0 .. c0 + 3 of the sample at xb
  __device__ __forceinline__ void window_task(const float* xb, float2 st, int pos0, int row0, int c0,
                                              uint8_t* win) const {
    const bool vec = (L & 3) == 0 && pos0 >= 0 && pos0 + 3 < L;  // whole float4s inside the row
    float4 xv[4], gv[4], bv[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int ci = c0 + c;
      xv[c] = gv[c] = bv[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ci < C) {
        const int64_t o = int64_t(ci) * L + pos0;
        if (vec) {
          xv[c] = __ldg(reinterpret_cast<const float4*>(xb + o));
          gv[c] = __ldg(reinterpret_cast<const float4*>(gamma + o));
          bv[c] = __ldg(reinterpret_cast<const float4*>(beta + o));
        } else {
          float e[3][4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const bool in = pos0 + i >= 0 && pos0 + i < L;
            e[0][i] = in ? __ldg(xb + o + i) : 0.f;
            e[1][i] = in ? __ldg(gamma + o + i) : 0.f;
            e[2][i] = in ? __ldg(beta + o + i) : 0.f;
          }
          xv[c] = make_float4(e[0][0], e[0][1], e[0][2], e[0][3]);
          gv[c] = make_float4(e[1][0], e[1][1], e[1][2], e[1][3]);
          bv[c] = make_float4(e[2][0], e[2][1], e[2][2], e[2][3]);
        }
      }
    }
    float a[4][4];  // [position][channel]
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const bool cin = c0 + c < C;
      const float xs[4] = {xv[c].x, xv[c].y, xv[c].z, xv[c].w}, gs[4] = {gv[c].x, gv[c].y, gv[c].z, gv[c].w},
                  bs[4] = {bv[c].x, bv[c].y, bv[c].z, bv[c].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool in = cin && pos0 + i >= 0 && pos0 + i < L;
        a[i][c] = in ? act(fmaf((xs[i] - st.x) * st.y, gs[i], bs[i])) : 0.f;
      }
    }
    const int q = (c0 & 31) >> 2;  // the 16-byte chunk of the channels
#pragma unroll
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4*>(win + chunk_off(row0 + i, q)) = make_float4(a[i][0], a[i][1], a[i][2], a[i][3]);
  }

  template <class Op>
  __device__ void convert(const ConvCtx& c) const {
    static_assert(Op::kind == MmaKind::TF32 && Op::kProducts == 3, "the fused path is the 3xTF32 mode");
    constexpr uint32_t kFull = 0xffffffffu;
    constexpr int kThreads = kConverterWarps * 32;
    const int ct = int(threadIdx.x) - kGemmThreads;  // 0 .. kThreads - 1
    const int lane = ct & 31;
    const bool copier = ct < 128;                     // A row ct of each stage
    uint8_t* win = c.scratch;
    int stage = 0;
    uint32_t phase = 0;
    for (int t = blockIdx.x; t < c.num_tiles; t += gridDim.x) {
      const Tile tl = tile(t);
      const float2 st = stats[tl.b];
      const float* xb = x + size_t(tl.b) * size_t(C) * size_t(L);
      const int l0 = tl.r0 - pad;          // the first position any tap reads
      const int la = (l0 >> 2) << 2;       // rounded down to a multiple of 4 (floor, also for l0 < 0)
      const int shift = l0 - la;
      const int quads = (wrows + shift + 3) >> 2;
      for (int cb = 0; cb < ncb; ++cb) {
        bar_sync(1, kThreads);  // the previous block's copies are done with the window
        for (int task = ct; task < quads * 8; task += kThreads) {
          const int qd = task >> 3, cq = task & 7;  // position quad, channel quartet
          window_task(xb, st, la + 4 * qd, 4 * qd, cb * 32 + 4 * cq, win);
        }
        bar_sync(1, kThreads);  // the window is complete
        if (!copier) continue;
        for (int tap = 0; tap < ksize; ++tap) {
          if (__any_sync(kFull, *c.abort_flag)) return;
          if (!__all_sync(kFull, mbar_wait<true>(&c.empty[stage], phase ^ 1))) {
            record_error(c.status, GF_DEV_WAIT_TIMEOUT);
            *c.abort_flag = 1;
            return;
          }
          uint8_t* a_hi = c.stages + stage * c.stage_bytes;
          uint8_t* a_lo = a_hi + c.a_bytes / 2;
          const int src_row = ct + shift + tap * dil;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 h = *reinterpret_cast<const float4*>(win + chunk_off(src_row, q));
            const uint32_t off = chunk_off(ct, q);
            *reinterpret_cast<float4*>(a_hi + off) = h;
            *reinterpret_cast<float4*>(a_lo + off) =
                make_float4(h.x - tf32_hi(h.x), h.y - tf32_hi(h.y), h.z - tf32_hi(h.z), h.w - tf32_hi(h.w));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&c.full[stage]);
          if (++stage == c.nstages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  }
};

// Epilogue: out[b][co][j] = acc + conv_b[co] + x[b][co][j].
struct EpiConvResidual {
  static constexpr bool kFixedBN = true;
  struct Params {
    const float* conv_b;  // may be null
    const float* x;
    float* out;
    int C, L;
  };
  template <int BN>
  __device__ __forceinline__ static void apply(const Params& p, uint32_t taddr, const Tile& t, int row) {
    const int j = t.r0 + row;
    const bool valid = j < p.L;
#pragma unroll 1
    for (int g = 0; g < BN / 64; ++g) {
      const int n0 = t.n0 + g * 64;
      if (n0 >= p.C) break;  // uniform across the warp
      float v[64];
      tmem_load64(taddr + uint32_t(g * 64), v);
      const size_t base = (size_t(t.b) * p.C + n0) * size_t(p.L) + size_t(j);
      if (valid) {
        // All residual loads of a 32-column half are issued before any store:
        // out and x may alias as far as the compiler knows, so interleaving
        // them would serialise one DRAM latency per column.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float r[32];
#pragma unroll
          for (int c = 0; c < 32; ++c)
            r[c] = (n0 + 32 * h + c < p.C) ? __ldcs(p.x + base + size_t(32 * h + c) * p.L) : 0.f;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int co = n0 + 32 * h + c;
            if (co < p.C) {
              const float bias = p.conv_b ? __ldg(p.conv_b + co) : 0.f;
              __stcs(p.out + base + size_t(32 * h + c) * p.L, v[32 * h + c] + bias + r[c]);
            }
          }
        }
      }
    }
  }
};

namespace {
constexpr int kBNConv = 256;

bool conv_mode_ok(int32_t mode) {
  return mode == GF_MODE_FP32_3XTF32 || mode == GF_MODE_BF16 || mode == GF_MODE_FP32_3XBF16;
}

// bytes per element of all operand planes together
size_t plane_bytes(int32_t mode) { return mode == GF_MODE_FP32_3XTF32 ? 8 : (mode == GF_MODE_BF16 ? 2 : 4); }

// Input channels padded to a whole number of k-blocks (32 fp32 or 64 bf16
// channels), so that no k-block straddles two taps.
int64_t padded_channels(int64_t C, int32_t mode) {
  const int64_t q = mode == GF_MODE_FP32_3XTF32 ? 32 : 64;
  return (C + q - 1) / q * q;
}

struct ConvWs {
  size_t part, stats, a_planes, w_planes, total;
  int chunks;
  bool fused;  // the single GEMM with converter warps: no activation planes
};

// The fused LayerNorm/GELU/Conv1d GEMM (GF_FLAG_FUSED_PRODUCER) runs in the
// 3xTF32 mode when the taps' window (128 + (ksize - 1) dilation positions)
// fits its scratch.
bool conv_fused_fits(int64_t ksize, int64_t dilation) {
  return (ksize - 1) * dilation <= LnConvSrc<false>::kMaxWindow - 128;
}

ConvWs conv_ws(int64_t B, int64_t C, int64_t L, int64_t ksize, int32_t mode, bool fused) {
  const int64_t Cp = padded_channels(C, mode);
  ConvWs w{};
  w.fused = fused;
  w.chunks = int((C * L + kLnChunk - 1) / kLnChunk);
  size_t off = 0;
  w.part = off;
  off += align_up(size_t(B) * w.chunks * sizeof(double2), 256);
  w.stats = off;
  off += align_up(size_t(B) * sizeof(float2), 256);
  w.a_planes = off;
  // (3xTF32: the raw plane only when the GEMM computes the lo plane itself)
  const size_t act_bytes = mode == GF_MODE_FP32_3XTF32 && (kLoConv & 1) ? 4 : plane_bytes(mode);
  if (!fused) off += align_up(size_t(B) * L * Cp * act_bytes, 256);
  w.w_planes = off;
  off += align_up(size_t(C) * ksize * Cp * plane_bytes(mode), 256);
  w.total = off;
  return w;
}

// B = 0 (an empty batch) passes: the entry point then returns GF_OK without
// launching anything.
gf_status check_conv_shape(int64_t B, int64_t C, int64_t L, int64_t ksize, int32_t mode) {
  if (B < 0 || C < 1 || L < 1 || ksize < 1 || ksize > 16) return GF_ERR_SHAPE;
  (void)mode;  // any C: the operand planes pad the channels to whole k-blocks
  if (C > 1024) return GF_ERR_SHAPE;
  if (B > 65535 || L > (int64_t(1) << 30)) return GF_ERR_SHAPE;
  return GF_OK;
}

template <int MODE>
void launch_conv_prepass(const float* x, const float* ln_gamma, const float* ln_beta, const float2* stats,
                         void* a_planes, int64_t B, int64_t C, int64_t L, bool tanh_gelu, cudaStream_t s) {
  const int64_t Cp = padded_channels(C, MODE);
  const dim3 grid(unsigned((L + 127) / 128), unsigned(Cp / 32), unsigned(B));
  const int c = int(C), cp = int(Cp), l = int(L), b = int(B);
  const bool vec = L % 4 == 0;
  if (tanh_gelu && vec)
    ln_apply_gelu_split_kernel<MODE, true, true><<<grid, 256, 0, s>>>(x, ln_gamma, ln_beta, stats, a_planes, c, cp, l, b);
  else if (tanh_gelu)
    ln_apply_gelu_split_kernel<MODE, true, false><<<grid, 256, 0, s>>>(x, ln_gamma, ln_beta, stats, a_planes, c, cp, l,
                                                                       b);
  else if (vec)
    ln_apply_gelu_split_kernel<MODE, false, true><<<grid, 256, 0, s>>>(x, ln_gamma, ln_beta, stats, a_planes, c, cp, l,
                                                                       b);
  else
    ln_apply_gelu_split_kernel<MODE, false, false><<<grid, 256, 0, s>>>(x, ln_gamma, ln_beta, stats, a_planes, c, cp,
                                                                        l, b);
}

// The LayerNorm statistics' finalize and the weight split, in one launch.
template <int MODE>
void launch_finalize_weights(const float* x, const double2* part, float2* stats, int64_t B, int64_t C, int64_t L,
                             int chunks, float eps, const float* conv_w, void* w_planes, int32_t ksize,
                             const DeviceInfo& dev, cudaStream_t s) {
  const int64_t Cp = padded_channels(C, MODE);
  const int64_t n = C * Cp * ksize;
  const int64_t wblocks = (n + 255) / 256 < dev.sm_count * 4 ? (n + 255) / 256 : dev.sm_count * 4;
  ln_finalize_weights_kernel<MODE><<<unsigned(B + wblocks), 256, 0, s>>>(x, part, stats, C * L, chunks, eps, int(B),
                                                                         conv_w, w_planes, int(C), int(Cp), ksize);
}

template <class Op>
gf_status launch_conv_gemm(const DeviceInfo& dev, const void* a_planes, const void* w_planes, int64_t B, int64_t C,
                           int64_t L, int32_t ksize, int32_t dilation, int32_t padding,
                           const EpiConvResidual::Params& ep, cudaStream_t s) {
  OperandMaps maps{};
  const int64_t Cp = padded_channels(C, Op::kElem == 4 ? GF_MODE_FP32_3XTF32 : GF_MODE_BF16);
  const uint64_t da[3] = {uint64_t(Cp), uint64_t(L), uint64_t(B)};
  const uint32_t ba[3] = {uint32_t(Op::kBK), uint32_t(kBM), 1};
  const uint64_t db[2] = {uint64_t(ksize) * Cp, uint64_t(C)};
  const uint32_t bb[2] = {uint32_t(Op::kBK), uint32_t(kBNConv)};
  const size_t a_plane = size_t(B) * L * Cp * Op::kElem, w_plane = size_t(C) * ksize * Cp * Op::kElem;
  constexpr int LO = std::is_same<Op, OpTF32x3>::value ? kLoConv : 0;
  for (int p = 0; p < Op::kPlanes; ++p) {
    gf_status st = GF_OK;
    if (p == 0 || !(LO & 1))
      st = make_tmap(&maps.a[p], static_cast<const uint8_t*>(a_planes) + p * a_plane, Op::kElem, 3, da, ba);
    if (st != GF_OK) return st;
    if (p == 0 || !(LO & 2))
      st = make_tmap(&maps.b[p], static_cast<const uint8_t*>(w_planes) + p * w_plane, Op::kElem, 2, db, bb);
    if (st != GF_OK) return st;
  }
  using Src = ConvSrcT<LO>;
  Src src;
  src.C = int(Cp);  // channels per tap along K
  src.pad = padding;
  src.dil = dilation;
  src.ksize = ksize;
  src.num_jb = int((L + kBM - 1) / kBM);
  src.num_nb = int((C + kBNConv - 1) / kBNConv);
  src.num_kb = int(ksize * Cp / Op::kBK);
  src.kb_chunk = src.num_kb;
  src.bn = kBNConv;
  src.bk = Op::kBK;
  src.nsamples = int(B);
  const int64_t tiles = int64_t(B) * src.num_jb * src.num_nb;
  return launch_gemm<kBNConv, Op, Src, EpiConvResidual>(dev, maps, src, tiles, ep, s);
}
// The fused LayerNorm -> GELU -> dilated Conv1d GEMM (3xTF32): weight planes
// in the channel-block-major k order, A built by the converter warps.
template <bool TANH>
gf_status launch_conv_fused(const DeviceInfo& dev, const float* x, const float* ln_gamma, const float* ln_beta,
                            const float2* stats, const float* w_planes, int64_t B, int64_t C, int64_t L,
                            int32_t ksize, int32_t dilation, int32_t padding, const EpiConvResidual::Params& ep,
                            cudaStream_t s) {
  using Op = OpTF32x3;
  OperandMaps maps{};
  const int64_t Cp = padded_channels(C, GF_MODE_FP32_3XTF32);
  const uint64_t db[2] = {uint64_t(ksize) * Cp, uint64_t(C)};
  const uint32_t bb[2] = {uint32_t(Op::kBK), uint32_t(kBNConv)};
  const size_t w_plane = size_t(C) * ksize * Cp;
  for (int p = 0; p < Op::kPlanes; ++p) {
    const gf_status st = make_tmap(&maps.b[p], w_planes + p * w_plane, Op::kElem, 2, db, bb);
    if (st != GF_OK) return st;
  }
  LnConvSrc<TANH> src{};
  src.x = x;
  src.gamma = ln_gamma;
  src.beta = ln_beta;
  src.stats = stats;
  src.C = int(C);
  src.Cp = int(Cp);
  src.L = int(L);
  src.pad = padding;
  src.dil = dilation;
  src.ksize = ksize;
  src.num_jb = int((L + kBM - 1) / kBM);
  src.num_nb = int((C + kBNConv - 1) / kBNConv);
  src.num_kb = int(ksize * Cp / Op::kBK);
  src.bn = kBNConv;
  src.bk = Op::kBK;
  src.nsamples = int(B);
  src.kb_chunk = src.num_kb;
  src.ncb = int(Cp / 32);
  src.wrows = 128 + (ksize - 1) * dilation;
  const int64_t tiles = int64_t(B) * src.num_jb * src.num_nb;
  return launch_gemm<kBNConv, Op, LnConvSrc<TANH>, EpiConvResidual>(dev, maps, src, tiles, ep, s);
}
}  // namespace
}  // namespace gf

using namespace gf;

extern "C" {

size_t gf_ln_gelu_dconv1d_res_workspace_size(int64_t B, int64_t C, int64_t L, int32_t ksize, int32_t dilation,
                                             int32_t mode) {
  if (mode & ~(GF_FLAG_GELU_TANH | GF_FLAG_FUSED_PRODUCER | 0xff)) return 0;
  const bool fused = (mode & GF_FLAG_FUSED_PRODUCER) != 0;
  mode &= 0xff;
  if (!conv_mode_ok(mode) || check_conv_shape(B, C, L, ksize, mode) != GF_OK || B == 0 || dilation < 1) return 0;
  if (fused && (mode != GF_MODE_FP32_3XTF32 || !conv_fused_fits(ksize, dilation))) return 0;
  return conv_ws(B, C, L, ksize, mode, fused).total;
}

gf_status gf_ln_gelu_dconv1d_res(const float* x, const float* ln_gamma, const float* ln_beta, const float* conv_w,
                                 const float* conv_b, float* out, int64_t B, int64_t C, int64_t L, int32_t ksize,
                                 int32_t dilation, int32_t padding, float eps, int32_t mode, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  // (an empty batch, B = 0, may pass NULL for x and out)
  if ((B && (!x || !out)) || !ln_gamma || !ln_beta || !conv_w) return GF_ERR_NULL;
  if (mode & ~(GF_FLAG_GELU_TANH | GF_FLAG_FUSED_PRODUCER | 0xff)) return GF_ERR_MODE;
  const bool tanh_gelu = (mode & GF_FLAG_GELU_TANH) != 0;
  const bool fused = (mode & GF_FLAG_FUSED_PRODUCER) != 0;
  mode &= 0xff;
  if (!conv_mode_ok(mode) || (fused && mode != GF_MODE_FP32_3XTF32)) return GF_ERR_MODE;
  gf_status st = check_conv_shape(B, C, L, ksize, mode);
  if (st != GF_OK) return st;
  if (dilation < 1 || padding < 0 || int64_t(2) * padding != int64_t(dilation) * (ksize - 1)) return GF_ERR_SHAPE;
  if (int64_t(dilation) * (ksize - 1) > (int64_t(1) << 30)) return GF_ERR_SHAPE;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return GF_ERR_SHAPE;
  if (fused && !conv_fused_fits(ksize, dilation)) return GF_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(ln_gamma) || !aligned16(ln_beta) || !aligned16(conv_w) || !aligned16(out) ||
      (conv_b && !aligned16(conv_b)) || !aligned16(workspace))
    return GF_ERR_ALIGN;
  if (B == 0) return GF_OK;
  const ConvWs wl = conv_ws(B, C, L, ksize, mode, fused);
  if (!workspace) return GF_ERR_NULL;
  if (workspace_bytes < wl.total) return GF_ERR_WORKSPACE;
  const size_t xb = size_t(B) * C * L * 4;
  const Span ins[] = {{x, xb},
                      {ln_gamma, size_t(C) * L * 4},
                      {ln_beta, size_t(C) * L * 4},
                      {conv_w, size_t(C) * C * ksize * 4},
                      {conv_b, size_t(C) * 4},
                      {workspace, wl.total}};
  st = check_no_alias(Span{out, xb}, ins, 6);
  if (st != GF_OK) return st;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != GF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  double2* part = reinterpret_cast<double2*>(ws + wl.part);
  float2* stats = reinterpret_cast<float2*>(ws + wl.stats);
  void* a_planes = ws + wl.a_planes;
  void* w_planes = ws + wl.w_planes;

  if ((C * L) % 4 == 0)
    ln_partial_kernel<true><<<dim3(unsigned(wl.chunks), unsigned(B)), 256, 0, s>>>(x, part, C * L, wl.chunks);
  else
    ln_partial_kernel<false><<<dim3(unsigned(wl.chunks), unsigned(B)), 256, 0, s>>>(x, part, C * L, wl.chunks);
  switch (mode) {
    case GF_MODE_FP32_3XTF32:
      launch_finalize_weights<GF_MODE_FP32_3XTF32>(x, part, stats, B, C, L, wl.chunks, eps, conv_w, w_planes, ksize,
                                                   dev, s);
      break;
    case GF_MODE_BF16:
      launch_finalize_weights<GF_MODE_BF16>(x, part, stats, B, C, L, wl.chunks, eps, conv_w, w_planes, ksize, dev, s);
      break;
    default:
      launch_finalize_weights<GF_MODE_FP32_3XBF16>(x, part, stats, B, C, L, wl.chunks, eps, conv_w, w_planes, ksize,
                                                   dev, s);
  }
  EpiConvResidual::Params ep{conv_b, x, out, int(C), int(L)};
  if (wl.fused) {
    // (the weights were split into the fused GEMM's k order above; LayerNorm
    // + GELU are applied inside the GEMM)
    if ((st = cuda_status(cudaGetLastError())) != GF_OK) return st;
    return tanh_gelu ? launch_conv_fused<true>(dev, x, ln_gamma, ln_beta, stats, static_cast<const float*>(w_planes),
                                               B, C, L, ksize, dilation, padding, ep, s)
                     : launch_conv_fused<false>(dev, x, ln_gamma, ln_beta, stats,
                                                static_cast<const float*>(w_planes), B, C, L, ksize, dilation,
                                                padding, ep, s);
  }
  switch (mode) {
    case GF_MODE_FP32_3XTF32:
      launch_conv_prepass<GF_MODE_FP32_3XTF32>(x, ln_gamma, ln_beta, stats, a_planes, B, C, L, tanh_gelu, s);
      break;
    case GF_MODE_BF16:
      launch_conv_prepass<GF_MODE_BF16>(x, ln_gamma, ln_beta, stats, a_planes, B, C, L, tanh_gelu, s);
      break;
    default:
      launch_conv_prepass<GF_MODE_FP32_3XBF16>(x, ln_gamma, ln_beta, stats, a_planes, B, C, L, tanh_gelu, s);
  }
  if ((st = cuda_status(cudaGetLastError())) != GF_OK) return st;
  switch (mode) {
    case GF_MODE_FP32_3XTF32:
      return launch_conv_gemm<OpTF32x3>(dev, a_planes, w_planes, B, C, L, ksize, dilation, padding, ep, s);
    case GF_MODE_BF16:
      return launch_conv_gemm<OpBF16x1>(dev, a_planes, w_planes, B, C, L, ksize, dilation, padding, ep, s);
    default:
      return launch_conv_gemm<OpBF16x3>(dev, a_planes, w_planes, B, C, L, ksize, dilation, padding, ep, s);
  }
}

}  // extern "C"
