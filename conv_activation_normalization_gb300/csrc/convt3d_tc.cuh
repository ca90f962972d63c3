// ConvTranspose3d(k 3, stride 2, pad 1) with the contraction on tcgen05.
//
// Phase form (see convt3d.cu): the 2x2x2 outputs of cell (qd, qh, qw) come
// from the 2x2x2 inputs at q..q+1, and every tap feeds exactly one output
// phase.  So per cell the transposed conv is a tiny dense product
//
//   Y[cell][phase*16 + co] = sum_k  A[cell][k] * B[phase*16 + co][k]
//   A[cell][pos*Cin + ci]   = x[n, ci, qd+a, qh+b, qw+c]   (pos = 4a + 2b + c)
//   B[(p)*16 + co][pos*Cin + ci] = w[ci, co, kd, kh, kw] when input offset a
//        feeds phase p in every dimension (a=0 -> k=1 for p=0, k=2 for p=1;
//        a=1 -> k=0 for p=1), else 0
//
// with K = 8 * Cin <= 32 (one 128-byte k-block), M = 128 cells per tile and
// N = 128 = 8 phases x 16 channels: a 128x128x32 3xTF32 MMA per tile (raw
// fp32 as hi, the tensor core truncates; lo = x - trunc(x)).  When K < 32 the
// conv bias rides in the padding: A[cell][K] = 1 and B[row][K] = bias[co].
//
// Roles (672 threads, one CTA per SM, persistent over tiles of 128 cells
// that run along the flattened (qh, qw) plane of one (n, qd)):
//   warps 0-3   producers: thread r gathers cell r's 8*Cin inputs and writes
//               the hi/lo rows of the A tile into an smem ring (128-byte
//               swizzle written by hand), fence.proxy.async, arrive;
//   warp 4      TMEM owner; one thread issues the 12 MMAs of a tile into one
//               of kCtTcAccBufs 128-column accumulators and commits;
//   warps 5-20  epilogue: warp (5 + e) reads TMEM lane quadrant (warp % 4)
//               and columns 32*(e / 4) .. +31 (output phases pd = e / 8,
//               ph = (e / 4) % 2, both pw), releases the accumulator, then
//                 PASS 1: Swish and per-group sums of s and s^2, reduced
//                         over the warp's 32 cells x 32 columns in fp32, one
//                         float2 per (sample, group, tile, warp), merged in
//                         fp64 by the finalize kernel;
//                 PASS 2: Swish, GroupNorm affine, HardSwish, stores.
// The weights tile B (hi/lo) is built once per CTA.
#pragma once

#include <cstdint>

#include "kernels_common.cuh"
#include "ptx.cuh"

namespace gf {

constexpr int kCtTcEpiWarps = 16;  // 4 per TMEM lane quadrant, 32 columns each
constexpr int kCtTcThreads = (5 + kCtTcEpiWarps) * 32;
constexpr int kCtTcProducerThreads = 128;
constexpr int kCtTcMmaWarp = 4;
constexpr int kCtTcEpiWarp0 = 5;
constexpr int kCtTcEpiThreads = kCtTcEpiWarps * 32;
constexpr int kCtTcStages = 4;
constexpr int kCtTcAccBufs = 2;  // TMEM accumulators of 128 columns
constexpr int kCtTcTmemCols = kCtTcAccBufs * 128 <= 256 ? 256 : 512;
constexpr int kCtTcPlane = 128 * 128;              // one 128-row x 128-byte tile
constexpr int kCtTcStageBytes = 2 * kCtTcPlane;    // A hi + lo
constexpr int kCtTcBBytes = 2 * kCtTcPlane;        // B hi + lo
constexpr int kCtTcSmem = kCtTcStages * kCtTcStageBytes + kCtTcBBytes + 1024 /*bars, scratch*/ + 1024 /*align*/;

// Division by a runtime constant as a multiply-shift (Granlund and
// Montgomery's round-up method): q = (umulhi(n, m) + n) >> l with
// l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1; exact for n < 2^31.
struct FastDiv {
  uint32_t d, m, l;
};

inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while ((uint64_t(1) << l) < d) ++l;
  const uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1;
  return FastDiv{d, uint32_t(m), l};
}

__device__ __forceinline__ int fdiv(int n, const FastDiv& f) {
  return int((__umulhi(uint32_t(n), f.m) + uint32_t(n)) >> f.l);
}

struct CtTcParams {
  const float* x;
  const float* w;
  const float* bias;     // may be null
  float2* part;          // PASS 1: [N][4][P][16] (sum s, sum s^2) per tile and epilogue warp
  const float2* coef;    // PASS 2: [N][16] (A, B)
  float* out;            // PASS 2
  int N, Cin, D, H, W;
  int bpp;               // tiles per (n, qd) plane: ceil(H*W / 128)
  int num_tiles;         // N * D * bpp
  FastDiv div_dp, div_bpp, div_w;  // by D * bpp, bpp and W
};

// tile t -> sample n, tile index within the sample rem, depth cell qd and the
// first flattened (qh, qw) cell index of the tile
struct CtTile {
  int n, rem, qd, c0;
};
__device__ __forceinline__ CtTile ct_tile(const CtTcParams& p, int t) {
  CtTile r;
  r.n = fdiv(t, p.div_dp);
  r.rem = t - r.n * int(p.div_dp.d);
  r.qd = fdiv(r.rem, p.div_bpp);
  r.c0 = (r.rem - r.qd * p.bpp) * 128;
  return r;
}

// byte offset of fp32 element k of row r in a K-major 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw128_offset(int r, int k) {
  return uint32_t(r) * 128u + ((uint32_t(k >> 2) ^ uint32_t(r & 7)) << 4) + uint32_t(k & 3) * 4u;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// phase p = pd*4 + ph*2 + pw exists for the cell
__device__ __forceinline__ bool ct_phase_ok(int p, int qd, int qh, int qw, int D, int H, int W) {
  return ((p >> 2) == 0 || qd < D - 1) && (((p >> 1) & 1) == 0 || qh < H - 1) && ((p & 1) == 0 || qw < W - 1);
}

template <int PASS, int CIN>
__global__ void __launch_bounds__(kCtTcThreads, 1) convt3d_tc_kernel(const CtTcParams p, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a_ring = smem;                                    // [S][hi, lo]
  uint8_t* b_tile = smem + kCtTcStages * kCtTcStageBytes;    // [hi, lo]
  uint64_t* full = reinterpret_cast<uint64_t*>(b_tile + kCtTcBBytes);
  uint64_t* empty = full + kCtTcStages;
  uint64_t* tfull = empty + kCtTcStages;
  uint64_t* tempty = tfull + kCtTcAccBufs;
  uint64_t* drain = tempty + kCtTcAccBufs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  constexpr int K = 8 * CIN;
  const int HW = p.H * p.W;

  // ---- setup: barriers, B tile, zero padding of the A ring, TMEM
  if (threadIdx.x == 0) {
    for (int s = 0; s < kCtTcStages; ++s) {
      mbar_init(&full[s], kCtTcProducerThreads);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < kCtTcAccBufs; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kCtTcEpiThreads);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < 128 * 32; i += blockDim.x) {
    const int row = i / 32, k = i % 32;  // row = phase*16 + co
    float v = 0.f;
    if (k == K && K < 32) {
      v = p.bias ? __ldg(p.bias + row % 16) : 0.f;  // the bias column (A holds 1 there)
    } else if (k < K) {
      const int pos = k / CIN, ci = k % CIN;
      const int ph3 = row / 16, co = row % 16;
      // per dimension d (depth, height, width = bit 2, 1, 0 of pos and ph3):
      // input offset a feeds phase: a=0 -> (p=0, k=1) or (p=1, k=2);
      // a=1 -> (p=1, k=0); (a=1, p=0) is no tap
      const int ad = (pos >> 2) & 1, ah = (pos >> 1) & 1, aw = pos & 1;
      const int pd_ = (ph3 >> 2) & 1, ph_ = (ph3 >> 1) & 1, pw_ = ph3 & 1;
      const bool used = (ad <= pd_) && (ah <= ph_) && (aw <= pw_);
      const int kd = ad ? 0 : (pd_ ? 2 : 1), kh = ah ? 0 : (ph_ ? 2 : 1), kw = aw ? 0 : (pw_ ? 2 : 1);
      const int tap = (kd * 3 + kh) * 3 + kw;
      if (used) v = __ldg(p.w + (size_t(ci) * 16 + co) * 27 + tap);
    }
    *reinterpret_cast<float*>(b_tile + sw128_offset(row, k)) = v;
    *reinterpret_cast<float*>(b_tile + kCtTcPlane + sw128_offset(row, k)) = v - tf32_hi(v);
  }
  // the K padding of every A row is written once: 1 in column K of the hi
  // plane (so the GEMM adds the bias column of B) and zeros elsewhere
  for (int i = threadIdx.x; i < kCtTcStages * 2 * 128 * 32; i += blockDim.x) {
    const int k = i % 32, row = (i / 32) % 128, plane = (i / (32 * 128)) & 1;
    if (k >= K)
      *reinterpret_cast<float*>(a_ring + (i / (32 * 128)) * kCtTcPlane + sw128_offset(row, k)) =
          (k == K && plane == 0) ? 1.f : 0.f;
  }
  fence_proxy_async_smem();
  if (warp == kCtTcMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kCtTcTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp < 4) {
    // ------------------------------------------------------------ producers
    const int r = threadIdx.x;  // cell row of the tile
    int stage = 0;
    uint32_t phase = 0;
    for (int t = blockIdx.x; t < p.num_tiles && !*abort_flag; t += gridDim.x) {
      const CtTile tl = ct_tile(p, t);
      const int n = tl.n, qd = tl.qd, c = tl.c0 + r;
      const bool cv = c < HW;
      const int qh = cv ? fdiv(c, p.div_w) : 0, qw = cv ? c - qh * p.W : 0;
      bool ok = mbar_wait<true>(&empty[stage], phase ^ 1);
      if (!ok) {
        record_error(status, GF_DEV_WAIT_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      // all gathers first (independent loads in flight together), then the
      // swizzled hi/lo rows of the A tile
      const bool vd = qd + 1 < p.D, vh = qh + 1 < p.H, vw = qw + 1 < p.W;
      const float* xc = p.x + (size_t(n) * CIN * p.D + qd) * HW + size_t(qh) * p.W + qw;
      float v[K];
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const int pos = k / CIN, ci = k % CIN;
        const int a = pos >> 2, b = (pos >> 1) & 1, c = pos & 1;
        const bool ok = cv && (a == 0 || vd) && (b == 0 || vh) && (c == 0 || vw);
        v[k] = ok ? __ldg(xc + size_t(ci) * p.D * HW + a * HW + b * p.W + c) : 0.f;
      }
      uint8_t* a_hi = a_ring + stage * kCtTcStageBytes;
      uint8_t* a_lo = a_hi + kCtTcPlane;
#pragma unroll
      for (int ch = 0; ch < K / 4; ++ch) {
        const float v0 = v[4 * ch], v1 = v[4 * ch + 1], v2 = v[4 * ch + 2], v3 = v[4 * ch + 3];
        const uint32_t off = sw128_offset(r, ch * 4);
        *reinterpret_cast<float4*>(a_hi + off) = make_float4(v0, v1, v2, v3);
        *reinterpret_cast<float4*>(a_lo + off) =
            make_float4(v0 - tf32_hi(v0), v1 - tf32_hi(v1), v2 - tf32_hi(v2), v3 - tf32_hi(v3));
      }
      fence_proxy_async_smem();
      mbar_arrive(&full[stage]);
      if (++stage == kCtTcStages) {
        stage = 0;
        phase ^= 1;
      }
    }
  } else if (warp == kCtTcMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_tf32(128, 128);
      const uint32_t b_hi = smem_u32(b_tile), b_lo = b_hi + kCtTcPlane;
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.num_tiles && ok && !*abort_flag; t += gridDim.x) {
        // the MMA thread polls: one thread costs few issue slots, and its
        // wake-up latency is on the critical path
        if (!(ok = mbar_wait(&tempty[acc], acc_phase ^ 1))) break;
        tc_fence_after();
        if (!(ok = mbar_wait(&full[stage], phase))) break;
        tc_fence_after();
        const uint32_t d = tmem_base + uint32_t(acc * 128);
        const uint32_t a_hi = smem_u32(a_ring + stage * kCtTcStageBytes), a_lo = a_hi + kCtTcPlane;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t off = uint32_t(kk * 32);
          mma_tf32(d, sdesc_kmajor_sw128(a_lo + off), sdesc_kmajor_sw128(b_hi + off), idesc, kk != 0);
          mma_tf32(d, sdesc_kmajor_sw128(a_hi + off), sdesc_kmajor_sw128(b_lo + off), idesc, 1u);
          mma_tf32(d, sdesc_kmajor_sw128(a_hi + off), sdesc_kmajor_sw128(b_hi + off), idesc, 1u);
        }
        mma_commit(&empty[stage]);
        mma_commit(&tfull[acc]);
        if (++stage == kCtTcStages) {
          stage = 0;
          phase ^= 1;
        }
        if (++acc == kCtTcAccBufs) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (!ok) {
        record_error(status, GF_DEV_WAIT_TIMEOUT);
        *abort_flag = 1;
      }
      mma_commit(drain);
      if (!mbar_wait<true>(drain, 0)) record_error(status, GF_DEV_WAIT_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - kCtTcEpiWarp0;  // 0..15
    const int quad = warp & 3, chunk = e >> 2;
    const int pd = chunk >> 1, hh = chunk & 1;  // depth and height phase of the chunk
    const int row = quad * 32 + lane;
    const int OD = 2 * p.D - 1, OH = 2 * p.H - 1, OW = 2 * p.W - 1;
    const int OHW = OH * OW;
    const size_t plane = size_t(OD) * OHW;
    const bool bias_in_epi = K == 32 && p.bias != nullptr;  // otherwise the GEMM added it
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      const CtTile tl = ct_tile(p, t);
      const int n = tl.n, rem = tl.rem, qd = tl.qd, c = tl.c0 + row;
      const bool cv = c < HW;
      const int qh = cv ? fdiv(c, p.div_w) : 0, qw = cv ? c - qh * p.W : 0;
      // GroupNorm coefficients of this sample, fetched before the wait: lane
      // co < 16 holds channel co's (A, B), read back with shuffles
      float2 abl = make_float2(0.f, 0.f);
      if constexpr (PASS == 2) abl = __ldg(p.coef + size_t(n) * 16 + (lane & 15));
      bool ok = __all_sync(0xffffffffu, mbar_wait<true>(&tfull[acc], acc_phase));
      if (!ok || *abort_flag) {
        if (!ok) {
          record_error(status, GF_DEV_WAIT_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      tc_fence_after();
      uint32_t r32[32];
      GF_TMEM_LD32(tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(acc * 128 + chunk * 32), r32);
      GF_TMEM_WAIT32(r32);
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (++acc == kCtTcAccBufs) {
        acc = 0;
        acc_phase ^= 1;
      }
      // columns (pw, co) of phase (pd, hh, pw); masks as 0/1 factors so no
      // branch separates the 32 Swish chains
      const bool pv0 = cv && ct_phase_ok(pd * 4 + hh * 2, qd, qh, qw, p.D, p.H, p.W);
      const bool pv1 = cv && ct_phase_ok(pd * 4 + hh * 2 + 1, qd, qh, qw, p.D, p.H, p.W);
      if constexpr (PASS == 1) {
        const float m0 = pv0 ? 1.f : 0.f, m1 = pv1 ? 1.f : 0.f;
        float gs[4] = {0.f, 0.f, 0.f, 0.f}, gq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int co = 0; co < 16; ++co) {
          const float b = bias_in_epi ? __ldg(p.bias + co) : 0.f;
          const float s0 = swish(__uint_as_float(r32[co]) + b) * m0;
          const float s1 = swish(__uint_as_float(r32[16 + co]) + b) * m1;
          gs[co >> 2] += s0 + s1;
          gq[co >> 2] = fmaf(s0, s0, fmaf(s1, s1, gq[co >> 2]));
        }
        // reduce-scatter of the 8 sums over the warp's 32 lanes (9 shuffles):
        // afterwards lane l holds the full sum of value v = 4*b4 + 2*b3 + b2
        // (b_i = bit i of l), value v being gs[v/2] (even v) or gq[v/2] (odd)
        float r[8] = {gs[0], gq[0], gs[1], gq[1], gs[2], gq[2], gs[3], gq[3]};
        {
          const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float send = b4 ? r[i] : r[4 + i];
            const float keep = b4 ? r[4 + i] : r[i];
            r[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
          }
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const float send = b3 ? r[i] : r[2 + i];
            const float keep = b3 ? r[2 + i] : r[i];
            r[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
          }
          {
            const float send = b2 ? r[0] : r[1];
            const float keep = b2 ? r[1] : r[0];
            r[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
          }
          r[0] += __shfl_xor_sync(0xffffffffu, r[0], 2);
          r[0] += __shfl_xor_sync(0xffffffffu, r[0], 1);
        }
        if ((lane & 3) == 0) {
          const int v = lane >> 2;  // 4*b4 + 2*b3 + b2
          float* dst = reinterpret_cast<float*>(p.part) +
                       (((size_t(n) * 4 + (v >> 1)) * size_t(p.D * p.bpp) + rem) * kCtTcEpiWarps + e) * 2 + (v & 1);
          *dst = r[0];
        }
      } else {
        float* ob = p.out + size_t(n) * 16 * plane + size_t((2 * qd + pd) * OHW + (2 * qh + hh) * OW + 2 * qw);
#pragma unroll
        for (int co = 0; co < 16; ++co) {
          const float b = bias_in_epi ? __ldg(p.bias + co) : 0.f;
          const float2 ab = make_float2(__shfl_sync(0xffffffffu, abl.x, co), __shfl_sync(0xffffffffu, abl.y, co));
          const float h0 = fmaf(ab.x, swish(__uint_as_float(r32[co]) + b), ab.y);
          const float h1 = fmaf(ab.x, swish(__uint_as_float(r32[16 + co]) + b), ab.y);
          float* oc = ob + size_t(co) * plane;
          if (pv0) __stcs(oc, h0 * __saturatef(fmaf(h0, 1.f / 6.f, 0.5f)));
          if (pv1) __stcs(oc + 1, h1 * __saturatef(fmaf(h1, 1.f / 6.f, 0.5f)));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kCtTcMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kCtTcTmemCols);
  }
}

}  // namespace gf
