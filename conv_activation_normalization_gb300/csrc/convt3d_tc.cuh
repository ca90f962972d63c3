// ConvTranspose3d(k 3, stride 2, pad 1) with the contraction on tcgen05.
//
// Phase form (see convt3d.cu): the 2x2x2 outputs of cell (qd, qh, qw) come
// from the 2x2x2 inputs at q..q+1, and every tap feeds exactly one output
// phase.  So per cell the transposed conv is a tiny dense product
//
//   Y[cell][col] = sum_k  A[cell][k] * B[col][k],  col = (pd*2 + ph)*32 + co*2 + pw
//   A[cell][pos*Cin + ci] = x[n, ci, qd+a, qh+b, qw+c]   (pos = 4a + 2b + c)
//   B[col][pos*Cin + ci]  = w[ci, co, kd, kh, kw] when input offset a feeds
//        phase p in every dimension (a=0 -> k=1 for p=0, k=2 for p=1;
//        a=1 -> k=0 for p=1), else 0
//
// The column order puts the two width phases of a channel side by side, so a
// 32-column slice of the accumulator is 16 (pw 0, pw 1) pairs that the
// epilogue processes with packed f32x2 arithmetic.
//
// with K = 8 * Cin <= 32 (one 128-byte k-block), M = 128 cells per tile and
// N = 128 = 8 phases x 16 channels: a 128x128x32 3xTF32 MMA per tile (raw
// fp32 as hi, the tensor core truncates; lo = x - trunc(x)).  When K < 32 the
// conv bias rides in the padding: A[cell][K] = 1 and B[row][K] = bias[co].
//
// Roles (5 + kCtTcEpiWarps warps, one CTA per SM, persistent over tiles of
// 128 cells that run along the flattened (qh, qw) plane of one (n, qd)):
//   warps 0-3   producers: thread r gathers cell r's 8*Cin inputs (coalesced
//               loads per warp, the neighbouring width position by shuffle)
//               and writes the hi and lo rows of a ring stage (128-byte
//               swizzle computed by hand), fence.proxy.async, and each warp
//               arrives once;
//   warp 4      TMEM owner; one thread issues the 12 MMAs of a tile into one
//               of kCtTcAccBufs 128-column accumulators and commits;
//   warps 5-    epilogue: warp (5 + e) reads TMEM lane quadrant (warp % 4)
//               and kCtTcEpiChunks chunks of 32 columns (chunk j = output
//               phases pd = j / 2, ph = j % 2, 16 channels x both pw), one
//               chunk at a time, releases the accumulator after the last
//               load, then
//                 PASS 1: Swish and per-group sums of s and s^2, reduced
//                         over the warp's 32 cells in fp32, one float2 per
//                         (sample, group, tile, warp), merged in fp64 by the
//                         finalize kernel;
//                 PASS 2: Swish, GroupNorm affine, HardSwish, stores.
// The weights tile B (hi/lo) is built once per CTA.
#pragma once

#include <cstdint>

#include "kernels_common.cuh"
#include "ptx.cuh"

namespace gf {

constexpr int kCtTcEpiWarps = 16;  // a multiple of 4 (one per TMEM lane quadrant)
constexpr int kCtTcEpiChunks = 16 / kCtTcEpiWarps;  // 32-column accumulator chunks per epilogue warp
constexpr int kCtTcThreads = (5 + kCtTcEpiWarps) * 32;
constexpr int kCtTcProducerThreads = 128;
constexpr int kCtTcMmaWarp = 4;
constexpr int kCtTcEpiWarp0 = 5;
constexpr int kCtTcEpiThreads = kCtTcEpiWarps * 32;
// operand stages: 3 (fused kernel on the 128-sample workload: 0.2283 ms
// against 0.2310 with 4 and 0.2382 with 2)
constexpr int kCtTcStages = 3;
constexpr int kCtTcAccBufs = 2;  // TMEM accumulators of 128 columns
constexpr int kCtTcTmemCols = kCtTcAccBufs * 128 <= 256 ? 256 : 512;
constexpr int kCtTcPlane = 128 * 128;              // one 128-row x 128-byte tile
constexpr int kCtTcStageBytes = 2 * kCtTcPlane;    // A hi + lo
constexpr int kCtTcBBytes = 2 * kCtTcPlane;        // B hi + lo
constexpr int kCtTcCoefBytes = kCtTcEpiWarps * 16 * 16;  // per epilogue warp: 16 channels x (A, A, B, B)
constexpr int kCtTcSmem =
    kCtTcStages * kCtTcStageBytes + kCtTcBBytes + kCtTcCoefBytes + 1024 /*bars, scratch*/ + 1024 /*align*/;

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
  const float4* coef;    // PASS 2: [N][16] (A, A, B, B)
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
template <class Prm>
__device__ __forceinline__ CtTile ct_tile(const Prm& p, int t) {
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

// phase p = pd*4 + ph*2 + pw exists for the cell
__device__ __forceinline__ bool ct_phase_ok(int p, int qd, int qh, int qw, int D, int H, int W) {
  return ((p >> 2) == 0 || qd < D - 1) && (((p >> 1) & 1) == 0 || qh < H - 1) && ((p & 1) == 0 || qw < W - 1);
}

// The weights tile B (hi/lo, rows in accumulator-column order), its values
// multiplied by `scale`, and the K padding of every A ring row: 1 in column K
// of the hi plane (so the GEMM adds the bias column of B, scaled too) and
// zeros elsewhere.  All threads of the CTA take part; the caller fences and
// synchronises.
template <int CIN>
__device__ __forceinline__ void ct_fill_tiles(const float* w, const float* bias, uint8_t* a_ring, uint8_t* b_tile,
                                              float scale = 1.f) {
  constexpr int K = 8 * CIN;
  for (int i = threadIdx.x; i < 128 * 32; i += blockDim.x) {
    const int row = i / 32, k = i % 32;  // row = (pd*2 + ph)*32 + co*2 + pw
    const int co = (row >> 1) & 15, ph3 = ((row >> 5) << 1) | (row & 1);
    float v = 0.f;
    if (k == K && K < 32) {
      v = bias ? __ldg(bias + co) : 0.f;  // the bias column (A holds 1 there)
    } else if (k < K) {
      const int pos = k / CIN, ci = k % CIN;
      // per dimension d (depth, height, width = bit 2, 1, 0 of pos and ph3):
      // input offset a feeds phase: a=0 -> (p=0, k=1) or (p=1, k=2);
      // a=1 -> (p=1, k=0); (a=1, p=0) is no tap
      const int ad = (pos >> 2) & 1, ah = (pos >> 1) & 1, aw = pos & 1;
      const int pd_ = (ph3 >> 2) & 1, ph_ = (ph3 >> 1) & 1, pw_ = ph3 & 1;
      const bool used = (ad <= pd_) && (ah <= ph_) && (aw <= pw_);
      const int kd = ad ? 0 : (pd_ ? 2 : 1), kh = ah ? 0 : (ph_ ? 2 : 1), kw = aw ? 0 : (pw_ ? 2 : 1);
      const int tap = (kd * 3 + kh) * 3 + kw;
      if (used) v = __ldg(w + (size_t(ci) * 16 + co) * 27 + tap);
    }
    v *= scale;
    *reinterpret_cast<float*>(b_tile + sw128_offset(row, k)) = v;
    *reinterpret_cast<float*>(b_tile + kCtTcPlane + sw128_offset(row, k)) = v - tf32_hi(v);
  }
  for (int i = threadIdx.x; i < kCtTcStages * 2 * 128 * 32; i += blockDim.x) {
    const int k = i % 32, row = (i / 32) % 128, plane = (i / (32 * 128)) & 1;
    if (k >= K)
      *reinterpret_cast<float*>(a_ring + (i / (32 * 128)) * kCtTcPlane + sw128_offset(row, k)) =
          (k == K && plane == 0) ? 1.f : 0.f;
  }
}

// Per-cell record of a tile for the output side of the single-kernel path
// (CtRecords): the element index of the cell's first output
// (n, co 0, 2 qd, 2 qh, 2 qw) in bits 0-55 and in bits 56-59 whether the cell
// exists (cv) and whether its second phase exists along depth (vd), height
// (vh) and width (vw).
constexpr int kCtRecSlots = 8;  // tiles whose records are kept (see convt3d_fused.cuh)
struct CtRecords {
  uint64_t* ring;     // [kCtRecSlots][128] in shared memory
  uint64_t* full;     // [kCtRecSlots] mbarriers: one arrival per producer warp
  uint64_t plane;     // output elements per (sample, channel)
  int OHW, OW;
};

// Producer warps 0-3: thread r gathers the 8 Cin inputs of cell r of the tile
// into row r of the A operand (hi = the raw values, lo = value - TF32 part),
// warp w holding 32 consecutive cells.  For each (ci, depth offset a, height
// offset b) every lane loads the input at its own width position qw (one
// coalesced load per warp) and takes the one at qw + 1 from the next lane,
// which holds cell (qh, qw + 1) whenever qw + 1 < W; the last lane loads it
// itself.  Inputs outside the volume are zero.  Once its 32 rows (and, with
// RECORDS, the cells' records) are written the warp arrives on the stage's
// full barrier (and the record slot's).
template <int CIN, bool RECORDS, class Prm>
__device__ __forceinline__ void ct_produce(const Prm& p, uint8_t* a_ring, uint64_t* full, uint64_t* empty,
                                           volatile uint32_t* abort_flag, uint32_t* status, const CtRecords& rec) {
  constexpr int K = 8 * CIN;
  constexpr uint32_t kFull = 0xffffffffu;
  const int lane = threadIdx.x % 32;
  const int r = threadIdx.x;  // cell row of the tile
  const int HW = p.H * p.W;
  const size_t sD = size_t(HW), sC = size_t(p.D) * sD;  // strides of a depth slice and an input channel
  int stage = 0, count = 0;
  uint32_t phase = 0;
  for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++count) {
    if (__any_sync(kFull, *abort_flag)) break;
    if (!__all_sync(kFull, mbar_wait<true>(&empty[stage], phase ^ 1))) {
      record_error(status, GF_DEV_WAIT_TIMEOUT);
      *abort_flag = 1;
      break;
    }
    const CtTile tl = ct_tile(p, t);
    const int n = tl.n, qd = tl.qd, c = tl.c0 + r;
    const bool cv = c < HW;
    const int qh = cv ? fdiv(c, p.div_w) : 0, qw = cv ? c - qh * p.W : 0;
    const bool vd = qd + 1 < p.D, vh = qh + 1 < p.H, vw = qw + 1 < p.W;
    const float* xb = p.x + (size_t(n) * CIN * p.D + qd) * sD + size_t(qh) * p.W + qw;
    float v[K];  // the A row in k order: k = pos * CIN + ci, pos = 4 a + 2 b + (width offset)
#pragma unroll
    for (int ci = 0; ci < CIN; ++ci)
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const bool ok = cv && (a == 0 || vd) && (b == 0 || vh);
          const float* src = xb + ci * sC + a * sD + b * p.W;
          const float v0 = ok ? __ldg(src) : 0.f;
          const float own = (ok && vw && lane == 31) ? __ldg(src + 1) : 0.f;
          const float nb = __shfl_down_sync(kFull, v0, 1);
          v[(4 * a + 2 * b) * CIN + ci] = v0;
          v[(4 * a + 2 * b + 1) * CIN + ci] = vw ? (lane == 31 ? own : nb) : 0.f;
        }
    uint8_t* a_hi = a_ring + stage * kCtTcStageBytes;
    uint8_t* a_lo = a_hi + kCtTcPlane;
#pragma unroll
    for (int ch = 0; ch < K / 4; ++ch) {
      const float4 h = make_float4(v[4 * ch], v[4 * ch + 1], v[4 * ch + 2], v[4 * ch + 3]);
      const uint32_t off = sw128_offset(r, ch * 4);
      *reinterpret_cast<float4*>(a_hi + off) = h;
      *reinterpret_cast<float4*>(a_lo + off) =
          make_float4(h.x - tf32_hi(h.x), h.y - tf32_hi(h.y), h.z - tf32_hi(h.z), h.w - tf32_hi(h.w));
    }
    if constexpr (RECORDS) {
      const uint64_t base = cv ? (uint64_t(n) * 16) * rec.plane + uint64_t(2 * qd) * uint64_t(rec.OHW) +
                                     uint64_t(2 * qh) * uint64_t(rec.OW) + uint64_t(2 * qw)
                               : 0;
      const uint64_t flags = uint64_t(cv) | (uint64_t(vd) << 1) | (uint64_t(vh) << 2) | (uint64_t(vw) << 3);
      rec.ring[(count % kCtRecSlots) * 128 + r] = base | (flags << 56);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&full[stage]);
      if constexpr (RECORDS) mbar_arrive(&rec.full[count % kCtRecSlots]);
    }
    if (++stage == kCtTcStages) {
      stage = 0;
      phase ^= 1;
    }
  }
}

// The MMA issuer (one thread): per tile the 3xTF32 MMAs of the k-steps of 8
// that hold data (the K = 8 Cin inputs, and the bias column when K < 32:
// lo x hi only where A's lo plane can be non-zero, k < K) into TMEM
// accumulator (tile count % NBUF), then commits to the ring stage's empty
// barrier and the accumulator's full barrier.
template <int NBUF, int CIN = 4, class Prm>
__device__ __forceinline__ void ct_mma(const Prm& p, uint32_t tmem_base, uint8_t* a_ring, uint8_t* b_tile,
                                       uint64_t* full, uint64_t* empty, uint64_t* tfull, uint64_t* tempty,
                                       uint64_t* drain, volatile uint32_t* abort_flag, uint32_t* status) {
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
    constexpr int K = 8 * CIN;
    constexpr int kSteps = K < 32 ? (K + 1 + 7) / 8 : 4;  // k-steps holding inputs or the bias column
    constexpr int kLoSteps = (K + 7) / 8;                // k-steps where A's lo plane can be non-zero
#pragma unroll
    for (int kk = 0; kk < kSteps; ++kk) {
      const uint32_t off = uint32_t(kk * 32);
      if (kk < kLoSteps)
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
    if (++acc == NBUF) {
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

template <int PASS, int CIN>
__global__ void __launch_bounds__(kCtTcThreads, 1) convt3d_tc_kernel(const CtTcParams p, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a_ring = smem;                                    // [S][hi, lo]
  uint8_t* b_tile = smem + kCtTcStages * kCtTcStageBytes;    // [hi, lo]
  float* coef_s = reinterpret_cast<float*>(b_tile + kCtTcBBytes);  // [epilogue warp][16][4]
  uint64_t* full = reinterpret_cast<uint64_t*>(b_tile + kCtTcBBytes + kCtTcCoefBytes);
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
      mbar_init(&full[s], kCtTcProducerThreads / 32);  // one arrival per producer warp
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < kCtTcAccBufs; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kCtTcEpiWarps);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  ct_fill_tiles<CIN>(p.w, p.bias, a_ring, b_tile);
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
    ct_produce<CIN, false>(p, a_ring, full, empty, abort_flag, status, CtRecords{});
  } else if (warp == kCtTcMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0)
      ct_mma<kCtTcAccBufs, CIN>(p, tmem_base, a_ring, b_tile, full, empty, tfull, tempty, drain, abort_flag, status);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - kCtTcEpiWarp0;
    const int quad = warp & 3;                       // TMEM lane quadrant of the warp
    const int chunk0 = (e >> 2) * kCtTcEpiChunks;    // first 32-column chunk of the warp
    const int row = quad * 32 + lane;
    const int OD = 2 * p.D - 1, OH = 2 * p.H - 1, OW = 2 * p.W - 1;
    const int OHW = OH * OW;
    const size_t plane = size_t(OD) * OHW;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      const CtTile tl = ct_tile(p, t);
      const int n = tl.n, rem = tl.rem, qd = tl.qd, c = tl.c0 + row;
      const bool cv = c < HW;
      const int qh = cv ? fdiv(c, p.div_w) : 0, qw = cv ? c - qh * p.W : 0;
      // GroupNorm coefficients of the tile's sample, fetched before the wait
      // (lane co < 16 holds channel co's (A, A, B, B))
      float4 cpre = make_float4(0.f, 0.f, 0.f, 0.f);
      if constexpr (PASS == 2) cpre = __ldg(p.coef + size_t(n) * 16 + (lane & 15));
      bool ok = __all_sync(0xffffffffu, mbar_wait<true>(&tfull[acc], acc_phase));
      if (!ok || __any_sync(0xffffffffu, *abort_flag)) {
        if (!ok) {
          record_error(status, GF_DEV_WAIT_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      tc_fence_after();
      float* cf = coef_s + e * 64;  // the warp's coefficient slot: 16 x (A, A, B, B) (pass 2)
      if constexpr (PASS == 2) {
        // the sync before the write keeps lanes still reading the previous
        // tile's values safe
        __syncwarp();
        if (lane < 16) reinterpret_cast<float4*>(cf)[lane] = cpre;
        __syncwarp();
      }
      float2 gs[4], gq[4];  // pass 1: per-group (sum s, sum s^2) of the thread, as pairs
#pragma unroll
      for (int g = 0; g < 4; ++g) gs[g] = gq[g] = make_float2(0.f, 0.f);
#pragma unroll 1
      for (int cc = 0; cc < kCtTcEpiChunks; ++cc) {
        const int chunk = chunk0 + cc, pd = chunk >> 1, hh = chunk & 1;  // depth and height phase
        uint32_t r32[32];
        GF_TMEM_LD32(tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(acc * 128 + chunk * 32), r32);
        GF_TMEM_WAIT32(r32);
        if (cc == kCtTcEpiChunks - 1) {  // the accumulator is fully read: release it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[acc]);
        }
        // r32[2 co + pw] is channel co at phase (pd, hh, pw); pv0 / pv1 say
        // whether the pw = 0 / 1 output lies inside the output volume
        const bool pv0 = cv && ct_phase_ok(pd * 4 + hh * 2, qd, qh, qw, p.D, p.H, p.W);
        const bool pv1 = cv && ct_phase_ok(pd * 4 + hh * 2 + 1, qd, qh, qw, p.D, p.H, p.W);
        if constexpr (PASS == 1) {
          // outputs outside the volume are zeroed before Swish (Swish(0) = 0),
          // so no branch separates the 16 pair chains
          const float2 m = make_float2(pv0 ? 1.f : 0.f, pv1 ? 1.f : 0.f);
#pragma unroll
          for (int co = 0; co < 16; ++co) {
            float2 y = make_float2(__uint_as_float(r32[2 * co]), __uint_as_float(r32[2 * co + 1]));
            if constexpr (K == 32) {  // no padding column: the bias is added here
              if (p.bias) {
                const float b = __ldg(p.bias + co);
                y = add2(y, make_float2(b, b));
              }
            }
            const float2 sv = swish2(mul2(y, m));
            gs[co >> 2] = add2(gs[co >> 2], sv);
            gq[co >> 2] = fma2(sv, sv, gq[co >> 2]);
          }
        } else {
          // GroupNorm affine A s + B, then HardSwish h sat(h / 6 + 1/2), on
          // (pw 0, pw 1) pairs; the pair's two outputs are adjacent in memory
          float* oc = p.out + size_t(n) * 16 * plane + size_t((2 * qd + pd) * OHW + (2 * qh + hh) * OW + 2 * qw);
#pragma unroll
          for (int co = 0; co < 16; ++co) {
            float2 y = make_float2(__uint_as_float(r32[2 * co]), __uint_as_float(r32[2 * co + 1]));
            if constexpr (K == 32) {
              if (p.bias) {
                const float b = __ldg(p.bias + co);
                y = add2(y, make_float2(b, b));
              }
            }
            const float4 ab = reinterpret_cast<const float4*>(cf)[co];  // (A, A, B, B), a broadcast read
            const float2 h = fma2(make_float2(ab.x, ab.y), swish2(y), make_float2(ab.z, ab.w));
            // (f32x2 FMAs have no saturating form)
            const float2 o = mul2(h, make_float2(__saturatef(fmaf(h.x, 1.f / 6.f, 0.5f)),
                                                 __saturatef(fmaf(h.y, 1.f / 6.f, 0.5f))));
            if (pv0) __stcs(oc, o.x);
            if (pv1) __stcs(oc + 1, o.y);
            oc += plane;
          }
        }
      }
      if (++acc == kCtTcAccBufs) {
        acc = 0;
        acc_phase ^= 1;
      }
      if constexpr (PASS == 1) {
        // reduce-scatter of the 8 sums over the warp's 32 lanes (9 shuffles):
        // afterwards lane l holds the full sum of value v = 4*b4 + 2*b3 + b2
        // (b_i = bit i of l), value v being gs[v/2] (even v) or gq[v/2] (odd)
        float r[8];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          r[2 * g] = gs[g].x + gs[g].y;
          r[2 * g + 1] = gq[g].x + gq[g].y;
        }
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
