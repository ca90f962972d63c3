// Persistent, warp-specialised tcgen05 GEMM with a 3xTF32 split, whose TMEM
// accumulator drains straight into a fused epilogue (the big intermediate
// never goes to HBM).
//
//   D[128 x BN] = sum_k  A_lo*B_hi + A_hi*B_lo + A_hi*B_hi     (fp32 accumulate)
//
// A and B arrive as hi/lo planes (hi = the fp32 value with its low 13
// mantissa bits cleared, i.e. exactly a TF32 number; lo = value - hi, exact in
// fp32), so each product of the split drops only the lo*lo term and the
// rounding of lo to TF32: about 2^-21 relative per product, against 2^-11 for a
// single TF32 product.
//
// Roles (one CTA per SM, 192 threads):
//   warp 0      one thread issues TMA loads of the four operand tiles of a
//               k-block into a ring of smem stages (full/empty mbarriers);
//   warp 1      owns the TMEM allocation; one thread issues tcgen05.mma into
//               one of two TMEM accumulators (BN columns each) and commits to
//               the stage's "empty" barrier and, per tile, to "tmem_full";
//   warps 2..5  the epilogue: each thread owns one accumulator row (TMEM lane),
//               reads it with tcgen05.ld and runs the fused epilogue, then
//               frees the accumulator ("tmem_empty") for the tile after next.
// The two accumulators let tile i's epilogue overlap tile i+1's mainloop.
//
// The operand source (a plain [rows, K] matrix, or the implicit-GEMM view of
// a dilated Conv1d) and the epilogue are template policies.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "ptx.cuh"

namespace gf {

constexpr int kBM = 128;        // tile rows = TMEM lanes
constexpr int kBK = 32;         // fp32 per k-block = one 128-byte swizzle row
constexpr int kGemmThreads = 192;
constexpr int kEpiThreads = 128;

template <int BN>
struct TileCfg {
  static constexpr int A_BYTES = kBM * kBK * 4;
  static constexpr int B_BYTES = BN * kBK * 4;
  static constexpr int STAGE_BYTES = 2 * (A_BYTES + B_BYTES);
  static constexpr int STAGES = (208 * 1024) / STAGE_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
  static_assert(STAGES >= 2, "need at least two smem stages");
  static_assert(TMEM_COLS == 32 || TMEM_COLS == 64 || TMEM_COLS == 128 || TMEM_COLS == 256 ||
                    TMEM_COLS == 512,
                "TMEM allocation must be a power of two >= 32 columns");
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN must be 64, 128, 192 or 256");
};

// One output tile: rows r0..r0+127 of sample b (b = 0 for a plain GEMM),
// columns n0..n0+BN-1 (n-block nb).
struct Tile {
  int b, r0, n0, nb;
};

// A = planes[2][M][K], B = planes[2][N][K]; tensor maps are 3-D
// {K, rows, plane} with a {32, rows-per-tile, 1} box and 128-byte swizzle.
struct LinearSrc {
  int num_mb, num_nb, num_kb, bn;
  int m_fastest;  // tile order: consecutive tiles share an n-block (1) or an m-block (0)
  __device__ __forceinline__ int num_tiles() const { return num_mb * num_nb; }
  __device__ __forceinline__ Tile tile(int t) const {
    int mb, nb;
    if (m_fastest) {
      mb = t % num_mb;
      nb = t / num_mb;
    } else {
      nb = t % num_nb;
      mb = t / num_nb;
    }
    return Tile{0, mb * kBM, nb * bn, nb};
  }
  __device__ __forceinline__ void load(const CUtensorMap* ta, const CUtensorMap* tb, uint64_t* bar,
                                       uint32_t a_hi, uint32_t a_lo, uint32_t b_hi, uint32_t b_lo,
                                       const Tile& t, int kb) const {
    const int k0 = kb * kBK;
    tma_load_3d(a_hi, ta, bar, k0, t.r0, 0);
    tma_load_3d(a_lo, ta, bar, k0, t.r0, 1);
    tma_load_3d(b_hi, tb, bar, k0, t.n0, 0);
    tma_load_3d(b_lo, tb, bar, k0, t.n0, 1);
  }
};

// Implicit GEMM of a stride-1 dilated Conv1d.  Rows are output positions j of
// one sample, columns are output channels, and the reduction index is
// k = tap * C + ci.  A = activation planes[2][B][L][C] (4-D map {C, L, B,
// plane}, box {32, 128, 1, 1}); the k-block (tap, ci0..ci0+31) of tile rows
// j0..j0+127 is the box at l = j0 - pad + tap * dil: rows outside [0, L) come
// back as zeros from the TMA unit, which is exactly the conv's zero padding.
// B = weight planes[2][Cout][ksize * C] (3-D map).
struct ConvSrc {
  int C, pad, dil;
  int num_jb, num_nb, num_kb, bn, nsamples;
  __device__ __forceinline__ int num_tiles() const { return nsamples * num_jb * num_nb; }
  __device__ __forceinline__ Tile tile(int t) const {
    const int nb = t % num_nb;
    const int r = t / num_nb;
    const int jb = r % num_jb;
    const int b = r / num_jb;
    return Tile{b, jb * kBM, nb * bn, nb};
  }
  __device__ __forceinline__ void load(const CUtensorMap* ta, const CUtensorMap* tb, uint64_t* bar,
                                       uint32_t a_hi, uint32_t a_lo, uint32_t b_hi, uint32_t b_lo,
                                       const Tile& t, int kb) const {
    const int k0 = kb * kBK;
    const int tap = k0 / C;
    const int ci0 = k0 - tap * C;
    const int l = t.r0 - pad + tap * dil;
    tma_load_4d(a_hi, ta, bar, ci0, l, t.b, 0);
    tma_load_4d(a_lo, ta, bar, ci0, l, t.b, 1);
    tma_load_3d(b_hi, tb, bar, k0, t.n0, 0);
    tma_load_3d(b_lo, tb, bar, k0, t.n0, 1);
  }
};

template <int BN, class Src, class Epi>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm3xtf32_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const Src src, const typename Epi::Params ep, uint32_t* status) {
  using Cfg = TileCfg<BN>;
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * Cfg::STAGE_BYTES);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiThreads);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_tiles = src.num_tiles();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_phase = 0;
      for (int t = blockIdx.x; t < num_tiles && !*abort_flag; t += gridDim.x) {
        const Tile tile = src.tile(t);
        for (int kb = 0; kb < src.num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1)) {
            record_error(status, GF_DEV_WAIT_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          const uint32_t base = smem_u32(smem + stage * Cfg::STAGE_BYTES);
          mbar_arrive_expect_tx(&full[stage], Cfg::STAGE_BYTES);
          src.load(&tmA, &tmB, &full[stage], base, base + Cfg::A_BYTES, base + 2 * Cfg::A_BYTES,
                   base + 2 * Cfg::A_BYTES + Cfg::B_BYTES, tile, kb);
          issued |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Never leave with a TMA write into this CTA's smem still in flight.
      for (int s = 0; s < S; ++s)
        if ((issued >> s) & 1u)
          if (!mbar_wait(&full[s], (issued_phase >> s) & 1u)) record_error(status, GF_DEV_WAIT_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_tf32(kBM, BN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok && !*abort_flag; t += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + uint32_t(acc * BN);
        for (int kb = 0; kb < src.num_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t base = smem_u32(smem + stage * Cfg::STAGE_BYTES);
          const uint32_t a_hi = base, a_lo = base + Cfg::A_BYTES;
          const uint32_t b_hi = base + 2 * Cfg::A_BYTES, b_lo = b_hi + Cfg::B_BYTES;
#pragma unroll
          for (int kk = 0; kk < kBK / 8; ++kk) {
            const uint32_t off = uint32_t(kk * 32);  // 8 tf32 = 32 bytes along K
            mma_tf32(d, sdesc_kmajor_sw128(a_lo + off), sdesc_kmajor_sw128(b_hi + off), idesc,
                     (kb | kk) != 0);
            mma_tf32(d, sdesc_kmajor_sw128(a_hi + off), sdesc_kmajor_sw128(b_lo + off), idesc, 1u);
            mma_tf32(d, sdesc_kmajor_sw128(a_hi + off), sdesc_kmajor_sw128(b_hi + off), idesc, 1u);
          }
          mma_commit(&empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (!ok) {
        record_error(status, GF_DEV_WAIT_TIMEOUT);
        *abort_flag = 1;
      }
      // Wait for every MMA this thread issued before TMEM can be released.
      mma_commit(drain);
      if (!mbar_wait(drain, 0)) record_error(status, GF_DEV_WAIT_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;  // TMEM lanes this warp may read: 32*quad ..
    const int row = quad * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      const Tile tile = src.tile(t);
      bool ok = mbar_wait(&tfull[acc], acc_phase);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok || *abort_flag) {
        if (!ok) {
          record_error(status, GF_DEV_WAIT_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(acc * BN);
      Epi::template apply<BN>(ep, taddr, tile, row);
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace gf
