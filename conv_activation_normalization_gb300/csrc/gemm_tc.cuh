// Persistent, warp-specialised tcgen05 GEMM whose TMEM accumulator drains
// straight into a fused epilogue (the big intermediate never goes to HBM).
//
// The contraction runs in one of three operand modes (MmaOp):
//   OpTF32x3  D = sum_k A_lo*B_hi + A_hi*B_lo + A_hi*B_hi, kind::tf32.
//             "hi" is the raw fp32 tensor itself: the tensor core reads only
//             the top 10 mantissa bits of an fp32 operand (it truncates), so
//             raw x acts exactly as hi = x with its 13 low mantissa bits
//             cleared; "lo" = x - hi (exact in fp32) is a plane written by a
//             pre-pass.  Each product drops only lo*lo and the rounding of lo
//             to TF32: about 2^-21 relative, against 2^-11 for one TF32
//             product.
//   OpBF16x3  the same three products with BF16 planes hi = bf16(x),
//             lo = bf16(x - hi), kind::f16 (twice the TF32 rate): about
//             2^-16 relative per product.
//   OpBF16x1  one BF16 product (the BF16 mode).
// All modes accumulate in fp32 in TMEM.
//
// Roles (one CTA per SM, 320 threads, plus a source's converter warps or the
// lo-plane warps below):
//   warp 0      one thread issues TMA loads of a k-block's operand tiles (one
//               or two planes of A and of B) into a ring of smem stages
//               (full/empty mbarriers);
//   warp 1      owns the TMEM allocation; one thread issues tcgen05.mma into
//               one of two TMEM accumulators (BN columns each), commits to the
//               stage's "empty" barrier and, per tile, to "tmem_full";
//   warps 2..9  the epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 (one
//               accumulator row per thread) and, for tiles of 128 or more
//               columns, half of the columns (warps 2..5 the first half,
//               6..9 the second), runs the fused epilogue on them, then frees
//               the accumulator ("tmem_empty") for the tile after next.  The
//               epilogue sees its half as a tile of BN / 2 columns starting at
//               n0 + half * BN / 2 with n-block index 2 nb + half.
// The two accumulators let tile i's epilogue overlap tile i+1's mainloop.
// Every smem row is 128 bytes (32 fp32 or 64 bf16 along K) with 128-byte
// swizzle, so one MMA K-step is always 32 bytes of the row.
//
// The operand source (a plain [rows, K] matrix, or the implicit-GEMM view of
// a dilated Conv1d) and the epilogue are template policies.  A source may
// build the A operand itself instead of loading it (kConverterWarps > 0):
// then warp 0 loads only B, and that many more warps (after the epilogue
// warps) write each stage's A planes with ordinary shared-memory stores
// (fence.proxy.async, then one arrival per warp on the stage's full
// barrier), using kScratchBytes of shared memory of their own.
//
// In-SM lo planes (OpTF32x3; Src::kLoInSm, bit 0 for A, bit 1 for B): the
// producer loads only the raw fp32 tile of that operand, and kSplitWarps more
// warps write lo = x - trunc_tf32(x) into the stage's lo plane before the
// MMAs read it.  Elementwise, so the lo tile takes the hi tile's layout as it
// is (the swizzle depends only on a byte's offset within the 1024-byte-aligned
// tile).  The raw tiles they convert complete on the stage's "loaded"
// barrier, which these warps wait on, the operand loaded whole (both planes,
// if any) on "full", where the MMA waits for it and for the warps' arrivals
// once the lo plane is written: the conversion of one operand overlaps the
// other's copy.  The operand then needs no lo plane in memory and no pre-pass
// to write it.
//
// Chunked accumulation (epi_chunked below): the tensor core adds
// each MMA's products into the fp32 accumulator with truncation, which over a
// long K loop of same-signed products (all-positive operands, say) becomes a
// bias that grows with K^2: -0.32 on sums of about 2048 at K = 8192, against
// an fp32 rounding error of about 1e-3.  Such epilogues take the tile's K loop
// in chunks of kb_chunk k-blocks, each accumulated from zero into the two
// TMEM accumulators in turn; the epilogue warps add each finished chunk into
// a running total kept in TMEM columns beside the accumulators (fp32 adds
// with round-to-nearest), so the bias grows only with K * chunk length, and
// hand the total of the earlier chunks to the epilogue with the last chunk.
// The accumulator of the next chunk fills while the last one is being added,
// as it does across tiles.  This needs BN + BN / halves <= ACC_STRIDE
// columns (160-column tiles: 240 of 256).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "host_common.h"
#include "ptx.cuh"

namespace gf {

constexpr int kBM = 128;  // tile rows = TMEM lanes
constexpr int kEpiWarps = 8;  // two per TMEM lane quadrant
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;
// column halves of a BN-wide tile served by separate epilogue warps
__host__ __device__ constexpr int epi_halves(int bn) { return bn >= 128 ? 2 : 1; }

enum class MmaKind { TF32, BF16 };

template <MmaKind K, int NPROD>
struct MmaOp {
  static constexpr MmaKind kind = K;
  static constexpr int kElem = K == MmaKind::TF32 ? 4 : 2;  // bytes per element
  static constexpr int kBK = 128 / kElem;                    // K elements per k-block
  static constexpr int kProducts = NPROD;
  static constexpr int kPlanes = NPROD == 3 ? 2 : 1;         // hi (+ lo) per operand
  static_assert(NPROD == 1 || NPROD == 3, "one product or the three-term split");
  template <int BN>
  __host__ __device__ static constexpr uint32_t idesc() {
    return K == MmaKind::TF32 ? idesc_tf32(kBM, BN) : idesc_bf16(kBM, BN);
  }
  __device__ __forceinline__ static void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    if constexpr (K == MmaKind::TF32)
      mma_tf32(d, a, b, idesc, acc);
    else
      mma_bf16(d, a, b, idesc, acc);
  }
};
using OpTF32x3 = MmaOp<MmaKind::TF32, 3>;
using OpBF16x3 = MmaOp<MmaKind::BF16, 3>;
using OpBF16x1 = MmaOp<MmaKind::BF16, 1>;

constexpr int kMaxDynSmem = 227 * 1024;  // dynamic shared memory one CTA may use

template <int BN, class Op, int EXTRA = 0>
struct TileCfg {
  static constexpr int A_BYTES = kBM * 128;  // one plane of a 128-row tile
  static constexpr int B_BYTES = BN * 128;
  static constexpr int STAGE_BYTES = Op::kPlanes * (A_BYTES + B_BYTES);
  static constexpr int BAR_BYTES = 256;
  static constexpr int EXTRA_BYTES = EXTRA;  // after the barriers
  // as many stages (up to 8) as fit beside the barriers, the source's and
  // the epilogue's scratch and the 1024-byte alignment slack in the 227 KB
  // of shared memory a CTA may use
  static constexpr int STAGES_FIT = (kMaxDynSmem - BAR_BYTES - 1024 - EXTRA) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  // two accumulators, each starting on a multiple of TMEM_COLS / 2
  static constexpr int TMEM_COLS = 2 * BN <= 128 ? 128 : (2 * BN <= 256 ? 256 : 512);
  static constexpr int ACC_STRIDE = TMEM_COLS / 2;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + EXTRA + 1024;
  static_assert(STAGES >= 2, "need at least two smem stages");
  static_assert(SMEM_BYTES <= kMaxDynSmem, "over the shared memory a CTA may use");
  static_assert(TMEM_COLS == 128 || TMEM_COLS == 256 || TMEM_COLS == 512,
                "TMEM allocation must be a power of two >= 32 columns");
  // epilogue halves of BN / 2 columns are read in pieces of 16
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN must be a multiple of 32 in [64, 256]");
};

// TMA descriptors of the operand planes: a[0]/b[0] = hi (or the only
// operand), a[1]/b[1] = lo (three-product modes); c = the fp32 output [M][N]
// in boxes of 32 rows x 16 columns, for epilogues that store through TMA
// (epi_tma_store).
struct OperandMaps {
  CUtensorMap a[2];
  CUtensorMap b[2];
  CUtensorMap c;
};

// Converter warps of a source (0: TMA loads A) and their shared scratch.
template <class Src, class = void>
struct SrcConv {
  static constexpr int warps = 0;
  static constexpr int arrivals = 0;
  static constexpr int scratch = 0;
};
template <class Src>
struct SrcConv<Src, decltype(void(Src::kConverterWarps))> {
  static constexpr int warps = Src::kConverterWarps;
  static constexpr int arrivals = Src::kArrivingWarps;  // converter warps that arrive on a stage's full barrier
  static constexpr int scratch = Src::kScratchBytes;
};
// Epilogues that can write their output as boxes of 32 rows x 16 fp32
// columns, staged in shared memory and sent by TMA stores (kTmaStore), do so
// in the one-plane operand mode.  There the MMAs are fast enough that the
// plain path's stores bound the kernel: a thread owns a row, so each warp
// store instruction touches 32 rows' cache lines.  (The three-product modes
// are bound by their MMAs, and their larger stages leave no room for the
// boxes.)
template <class Epi, class = void>
struct EpiTma {
  static constexpr bool value = false;
};
template <class Epi>
struct EpiTma<Epi, decltype(void(Epi::kTmaStore))> {
  static constexpr bool value = Epi::kTmaStore;
};
template <class Epi, class Op>
__host__ __device__ constexpr bool epi_tma_store() {
  return EpiTma<Epi>::value && Op::kPlanes == 1;
}
constexpr int kStoreBoxFloats = 32 * 16;  // 2 KB: a row is 64 bytes (64-byte swizzle)
template <class Epi, class Op>
__host__ __device__ constexpr int epi_smem_bytes() {
  // two box buffers per epilogue warp, 1024-byte aligned
  return epi_tma_store<Epi, Op>() ? 1024 + kEpiWarps * 2 * kStoreBoxFloats * 4 : 0;
}

// An epilogue warp's output path through TMA stores: its two box buffers
// (used in turn), the output's tensor map, the first output row of the
// warp's 32 rows, and the number of boxes the warp has stored so far.
struct BoxStore {
  float* buf;
  const CUtensorMap* map;
  int y;
  uint32_t n;
};

// Operands whose lo plane the kernel computes (bit 0: A, bit 1: B).
template <class Src, class = void>
struct SrcLo {
  static constexpr int mask = 0;
};
template <class Src>
struct SrcLo<Src, decltype(void(Src::kLoInSm))> {
  static constexpr int mask = Src::kLoInSm;
};
constexpr int kSplitWarps = 4;

template <class Src, class Epi, class Op, int BN>
__host__ __device__ constexpr int gemm_threads() {
  return kGemmThreads + 32 * (SrcConv<Src>::warps + (SrcLo<Src>::mask ? kSplitWarps : 0));
}

// What the converter warps of a source get from the kernel: the stage ring
// and its barriers, the abort flag and status word, and their scratch.
struct ConvCtx {
  uint8_t* stages;       // stage s at stages + s * stage_bytes: A planes, then B planes
  int stage_bytes, a_bytes, nstages;
  uint64_t* full;
  uint64_t* empty;
  volatile uint32_t* abort_flag;
  uint32_t* status;
  uint8_t* scratch;
  int num_tiles;
};

// One output tile: rows r0..r0+127 of sample b (b = 0 for a plain GEMM),
// columns n0..n0+BN-1 (n-block nb).
struct Tile {
  int b, r0, n0, nb;
};

// Whether the epilogue takes its accumulator in chunks (for this operand mode
// and BNW epilogue columns per thread): epilogues that declare
// chunked<Op, BNW>() and say so.
template <class Epi, class = void>
struct HasChunked {
  static constexpr bool value = false;
};
template <class Epi>
struct HasChunked<Epi, decltype(void(&Epi::template apply_last<64>))> {
  static constexpr bool value = true;
};
template <class Epi, class Op, int BN>
__host__ __device__ constexpr bool epi_chunked() {
  if constexpr (HasChunked<Epi>::value)
    return Epi::template chunked<Op>() && BN + BN / epi_halves(BN) <= TileCfg<BN, Op>::ACC_STRIDE;
  else
    return false;
}

// A = [M][K] planes (2-D maps {K, M}, box {BK, 128}), B = [N][K] planes.
// LO: operands whose lo plane the kernel computes (not loaded).
template <int LO>
struct LinearSrcT {
  static constexpr int kLoInSm = LO;
  int num_mb, num_nb, num_kb, bn, bk;
  int kb_chunk;   // k-blocks per accumulation chunk (chunked epilogues only)
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
  template <int PLANES>
  __device__ __forceinline__ void load(const OperandMaps& m, uint64_t* bar, const uint32_t* sa, const uint32_t* sb,
                                       const Tile& t, int kb) const {
    load_split<PLANES>(m, bar, bar, sa, sb, t, kb);
  }
  // A's planes complete on bar_a, B's on bar_b; the lo planes the kernel
  // computes (LO) are not loaded
  template <int PLANES>
  __device__ __forceinline__ void load_split(const OperandMaps& m, uint64_t* bar_a, uint64_t* bar_b,
                                             const uint32_t* sa, const uint32_t* sb, const Tile& t, int kb) const {
    const int k0 = kb * bk;
    // the copies of the tiles the kernel converts go first
    auto load_a = [&] {
#pragma unroll
      for (int p = 0; p < PLANES; ++p)
        if (p == 0 || !(LO & 1)) tma_load_2d(sa[p], &m.a[p], bar_a, k0, t.r0);
    };
    auto load_b = [&] {
#pragma unroll
      for (int p = 0; p < PLANES; ++p)
        if (p == 0 || !(LO & 2)) tma_load_2d(sb[p], &m.b[p], bar_b, k0, t.n0);
    };
    if (LO == 0) {  // (the planes of A and B in turn)
#pragma unroll
      for (int p = 0; p < PLANES; ++p) {
        tma_load_2d(sa[p], &m.a[p], bar_a, k0, t.r0);
        tma_load_2d(sb[p], &m.b[p], bar_b, k0, t.n0);
      }
    } else if (LO == 2) {
      load_b();
      load_a();
    } else {
      load_a();
      load_b();
    }
  }
  // Clusters of CL CTAs: unit q is the group of m-blocks CL mg .. CL mg +
  // CL - 1 at one n-block, and cluster CTA `rank` takes m-block CL mg + rank.
  // When CL does not divide the number of m-blocks, the last group's tiles
  // past M still run (their A rows load as zeros; the epilogue skips them):
  // each CTA has to load its slice of the B tile the group shares.
  template <int CL>
  __device__ __forceinline__ int num_groups() const {
    return (num_mb + CL - 1) / CL * num_nb;
  }
  template <int CL>
  __device__ __forceinline__ Tile tile_of_group(int q, uint32_t rank) const {
    const int num_mg = (num_mb + CL - 1) / CL;
    int mg, nb;
    if (m_fastest) {
      mg = q % num_mg;
      nb = q / num_mg;
    } else {
      nb = q % num_nb;
      mg = q / num_nb;
    }
    return Tile{0, (CL * mg + int(rank)) * kBM, nb * bn, nb};
  }
  __device__ __forceinline__ bool live(const Tile& t) const { return t.r0 < num_mb * kBM; }
  // This CTA's A tile, and slice `rank` of the group's B tile (rows
  // n0 + rank * bn / CL ..) multicast into every CTA's stage at the same
  // offset; each CTA's full barrier counts its A and all CL slices of B.
  template <int CL>
  __device__ __forceinline__ void load_group(const OperandMaps& m, uint64_t* bar, uint32_t sa, uint32_t sb,
                                             const Tile& t, int kb, uint32_t rank) const {
    const int k0 = kb * bk;
    tma_load_2d(sa, &m.a[0], bar, k0, t.r0);
    tma_load_2d_mc(sb + rank * uint32_t(bn / CL * 128), &m.b[0], bar, k0, t.n0 + int(rank) * (bn / CL),
                   uint16_t((1u << CL) - 1));
  }
};
using LinearSrc = LinearSrcT<0>;

// Implicit GEMM of a stride-1 dilated Conv1d.  Rows are output positions j of
// one sample, columns are output channels, and the reduction runs over blocks
// of BK channels (outer) and taps (inner): k-block kb = cb * ksize + tap
// covers channels cb * BK .. + BK - 1 of tap `tap`.  A = activation planes
// [B][L][C] (3-D maps {C, L, B}, box {BK, 128, 1}); the k-block of tile rows
// j0..j0+127 is the box at l = j0 - pad + tap * dil: rows outside [0, L) come
// back as zeros from the TMA unit, which is exactly the conv's zero padding.
// B = weight planes [Cout][ksize * C] in the same k order (2-D maps).  With
// the taps inner, the first touch of each row block (a DRAM read) comes every
// ksize-th k-block instead of in a run of C / BK at the start of the tile.
// LO: operands whose lo plane the kernel computes (not loaded).
template <int LO>
struct ConvSrcT {
  static constexpr int kLoInSm = LO;
  int C, pad, dil, ksize;
  int num_jb, num_nb, num_kb, bn, bk, nsamples;
  int kb_chunk;   // k-blocks per accumulation chunk (chunked epilogues only)
  __device__ __forceinline__ int num_tiles() const { return nsamples * num_jb * num_nb; }
  __device__ __forceinline__ Tile tile(int t) const {
    const int nb = t % num_nb;
    const int r = t / num_nb;
    const int jb = r % num_jb;
    const int b = r / num_jb;
    return Tile{b, jb * kBM, nb * bn, nb};
  }
  template <int PLANES>
  __device__ __forceinline__ void load(const OperandMaps& m, uint64_t* bar, const uint32_t* sa, const uint32_t* sb,
                                       const Tile& t, int kb) const {
    load_split<PLANES>(m, bar, bar, sa, sb, t, kb);
  }
  // A's planes complete on bar_a, B's on bar_b; the lo planes the kernel
  // computes (LO) are not loaded
  template <int PLANES>
  __device__ __forceinline__ void load_split(const OperandMaps& m, uint64_t* bar_a, uint64_t* bar_b,
                                             const uint32_t* sa, const uint32_t* sb, const Tile& t, int kb) const {
    const int k0 = kb * bk;
    const int cb = kb / ksize;
    const int tap = kb - cb * ksize;
    const int ci0 = cb * bk;
    const int l = t.r0 - pad + tap * dil;
    // the copies of the tiles the kernel converts go first
    auto load_a = [&] {
#pragma unroll
      for (int p = 0; p < PLANES; ++p)
        if (p == 0 || !(LO & 1)) tma_load_3d(sa[p], &m.a[p], bar_a, ci0, l, t.b);
    };
    auto load_b = [&] {
#pragma unroll
      for (int p = 0; p < PLANES; ++p)
        if (p == 0 || !(LO & 2)) tma_load_2d(sb[p], &m.b[p], bar_b, k0, t.n0);
    };
    if (LO == 0) {  // (the planes of A and B in turn)
#pragma unroll
      for (int p = 0; p < PLANES; ++p) {
        tma_load_3d(sa[p], &m.a[p], bar_a, ci0, l, t.b);
        tma_load_2d(sb[p], &m.b[p], bar_b, k0, t.n0);
      }
    } else if (LO == 2) {
      load_b();
      load_a();
    } else {
      load_a();
      load_b();
    }
  }
};
using ConvSrc = ConvSrcT<0>;

// lo = x - trunc_tf32(x) of a BYTES-long fp32 tile in shared memory, written
// at the same offsets of `lo`, by the kSplitWarps * 32 threads (thread ct):
// all of a thread's 16-byte loads first, then the arithmetic and the stores.
template <int BYTES>
__device__ __forceinline__ void split_lo_tile(const uint8_t* hi, uint8_t* lo, int ct) {
  constexpr int kThreads = kSplitWarps * 32;
  constexpr int kPer = BYTES / 16 / kThreads;
  static_assert(BYTES % (16 * kThreads) == 0, "whole 16-byte pieces per thread");
  float4 v[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) v[j] = reinterpret_cast<const float4*>(hi)[ct + j * kThreads];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const float4 x = v[j];
    const float4 r = make_float4(x.x - __uint_as_float(__float_as_uint(x.x) & 0xFFFFE000u),
                                 x.y - __uint_as_float(__float_as_uint(x.y) & 0xFFFFE000u),
                                 x.z - __uint_as_float(__float_as_uint(x.z) & 0xFFFFE000u),
                                 x.w - __uint_as_float(__float_as_uint(x.w) & 0xFFFFE000u));
    reinterpret_cast<float4*>(lo)[ct + j * kThreads] = r;
  }
}

// CL > 1: the grid is made of clusters of CL CTAs that take m-adjacent tiles
// of one n-block together (Src::tile_of_group) and share the B tile: each CTA
// loads a slice of it and multicasts it into every CTA's stage, so the B
// bytes read from L2 per tile drop CL-fold.  A stage is then free only when
// every CTA's MMAs have read it: each MMA commit arrives on the stage's empty
// barrier in every CTA.  (One-plane operands and unchunked epilogues only.)
template <int BN, class Op, class Src, class Epi, int CL>
__global__ void __launch_bounds__(gemm_threads<Src, Epi, Op, BN>(), 1)
    gemm_tc_kernel(const __grid_constant__ OperandMaps maps, const Src src, const typename Epi::Params ep,
                   uint32_t* status) {
  static_assert(CL == 1 || ((CL == 2 || CL == 4) && Op::kPlanes == 1 && SrcConv<Src>::warps == 0 &&
                             !epi_chunked<Epi, Op, BN>() && BN % (8 * CL) == 0),
                "clusters: one operand plane, TMA-loaded A, unchunked epilogue, whole 8-row B slices");
  constexpr uint16_t kClusterMask = uint16_t((1u << CL) - 1);
  constexpr int kConv = SrcConv<Src>::warps;
  constexpr int kLo = SrcLo<Src>::mask;
  static_assert(kLo == 0 || (Op::kind == MmaKind::TF32 && Op::kPlanes == 2 && kConv == 0 && CL == 1),
                "lo planes are computed in the SM from raw fp32 tiles only (3xTF32), by their own warps");
  // (kLo) bytes of a stage on "loaded" (the raw tiles converted here) and on
  // "full" (an operand loaded with both planes)
  constexpr uint32_t kLoLoadedTx =
      ((kLo & 1) ? TileCfg<BN, Op>::A_BYTES : 0) + ((kLo & 2) ? TileCfg<BN, Op>::B_BYTES : 0);
  constexpr uint32_t kLoFullTx =
      ((kLo & 1) ? 0 : 2 * TileCfg<BN, Op>::A_BYTES) + ((kLo & 2) ? 0 : 2 * TileCfg<BN, Op>::B_BYTES);
  using Cfg = TileCfg<BN, Op, SrcConv<Src>::scratch + epi_smem_bytes<Epi, Op>()>;
  constexpr int S = Cfg::STAGES;
  constexpr int P = Op::kPlanes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * Cfg::STAGE_BYTES);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* loaded = drain + 1;  // (kLo) the raw tiles the lo-plane warps convert have landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(loaded + S);
  static_assert((3 * S + 5) * 8 + 8 <= Cfg::BAR_BYTES, "barriers overflow their space");
  volatile uint32_t* abort_flag = tmem_slot + 1;
  uint8_t* scratch = smem + S * Cfg::STAGE_BYTES + Cfg::BAR_BYTES;  // the converters' (kConv > 0)
  float* boxes = reinterpret_cast<float*>(  // the epilogue's TMA-store boxes
      (reinterpret_cast<uintptr_t>(scratch + SrcConv<Src>::scratch) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // the TMA thread (and the converter warps), or the lo-plane warps
      mbar_init(&full[s], kLo ? kSplitWarps + (kLoFullTx ? 1 : 0) : 1 + SrcConv<Src>::arrivals);
      mbar_init(&empty[s], CL);  // the MMA commit of each CTA of the cluster
      mbar_init(&loaded[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128 * epi_halves(BN));  // every thread of the active epilogue warps
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int p = 0; p < P; ++p) {
      prefetch_tmap(&maps.a[p]);
      prefetch_tmap(&maps.b[p]);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CL > 1) cluster_sync_all();  // the other CTAs' barriers are initialised
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_tiles = src.num_tiles();
  // the persistent loop's units: tiles, or (CL > 1) groups of CL tiles, one
  // per CTA of a cluster
  uint32_t crank = 0;
  if constexpr (CL > 1) crank = cluster_ctarank();
  const int unit0 = int(blockIdx.x) / CL, unit_step = int(gridDim.x) / CL;
  int num_units = num_tiles;
  if constexpr (CL > 1) num_units = src.template num_groups<CL>();
  auto unit_tile = [&](int u) -> Tile {
    if constexpr (CL > 1)
      return src.template tile_of_group<CL>(u, crank);
    else
      return src.tile(u);
  };
  // k-blocks per accumulation chunk: the whole K loop unless the epilogue
  // adds chunks (both the MMA issuer and the epilogue count chunks with it)
  constexpr bool kChunked = epi_chunked<Epi, Op, BN>();
  const int kb_chunk = kChunked && src.kb_chunk > 0 ? src.kb_chunk : src.num_kb;

  // smem address of plane p of A / B in stage s
  auto a_addr = [&](int s, int p) { return smem_u32(smem + s * Cfg::STAGE_BYTES + p * Cfg::A_BYTES); };
  auto b_addr = [&](int s, int p) {
    return smem_u32(smem + s * Cfg::STAGE_BYTES + P * Cfg::A_BYTES + p * Cfg::B_BYTES);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_phase = 0;
      for (int u = unit0; u < num_units && !*abort_flag; u += unit_step) {
        const Tile tile = unit_tile(u);
        for (int kb = 0; kb < src.num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1)) {
            record_error(status, GF_DEV_WAIT_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          uint32_t sa[2], sb[2];
#pragma unroll
          for (int p = 0; p < P; ++p) {
            sa[p] = a_addr(stage, p);
            sb[p] = b_addr(stage, p);
          }
          if constexpr (kLo != 0) {
            // the raw tiles the lo-plane warps convert first (their copies
            // issued first), then an operand loaded whole
            mbar_arrive_expect_tx(&loaded[stage], kLoLoadedTx);
            if constexpr (kLoFullTx != 0) mbar_arrive_expect_tx(&full[stage], kLoFullTx);
            src.template load_split<P>(maps, (kLo & 1) ? &loaded[stage] : &full[stage],
                                       (kLo & 2) ? &loaded[stage] : &full[stage], sa, sb, tile, kb);
          } else {
            // bytes the TMA brings: the stage less the converters' A planes
            mbar_arrive_expect_tx(&full[stage], kConv ? P * Cfg::B_BYTES : Cfg::STAGE_BYTES);
            if constexpr (CL > 1)
              src.template load_group<CL>(maps, &full[stage], sa[0], sb[0], tile, kb, crank);
            else
              src.template load<P>(maps, &full[stage], sa, sb, tile, kb);
          }
          issued |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Never leave with a TMA write into this CTA's smem still in flight
      // (with CL > 1 that includes the other CTAs' multicast slices), nor
      // (CL > 1) with another CTA's MMA commit still to arrive on an empty
      // barrier here.
      for (int s = 0; s < S; ++s)
        if ((issued >> s) & 1u) {
          if (!mbar_wait(kLo ? &loaded[s] : &full[s], (issued_phase >> s) & 1u))
            record_error(status, GF_DEV_WAIT_TIMEOUT);
          if constexpr (kLo != 0 && kLoFullTx != 0)
            if (!mbar_wait(&full[s], (issued_phase >> s) & 1u)) record_error(status, GF_DEV_WAIT_TIMEOUT);
          if constexpr (CL > 1)
            if (!mbar_wait(&empty[s], (issued_phase >> s) & 1u)) record_error(status, GF_DEV_WAIT_TIMEOUT);
        }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = Op::template idesc<BN>();
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      // the MMAs of one k-block into accumulator d; the first of a chunk
      // overwrites it
      auto mma_kblock = [&](uint32_t d, bool chunk_start) {
        const uint32_t a_hi = a_addr(stage, 0), b_hi = b_addr(stage, 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t off = uint32_t(kk * 32);  // one MMA K-step = 32 bytes of the row
          const uint32_t accumulate = !chunk_start || kk != 0;
          if constexpr (Op::kProducts == 3) {
            const uint32_t a_lo = a_addr(stage, 1), b_lo = b_addr(stage, 1);
            Op::mma(d, sdesc_kmajor_sw128(a_lo + off), sdesc_kmajor_sw128(b_hi + off), idesc, accumulate);
            Op::mma(d, sdesc_kmajor_sw128(a_hi + off), sdesc_kmajor_sw128(b_lo + off), idesc, 1u);
            Op::mma(d, sdesc_kmajor_sw128(a_hi + off), sdesc_kmajor_sw128(b_hi + off), idesc, 1u);
          } else {
            Op::mma(d, sdesc_kmajor_sw128(a_hi + off), sdesc_kmajor_sw128(b_hi + off), idesc, accumulate);
          }
        }
        if constexpr (CL > 1)
          mma_commit_mc(&empty[stage], kClusterMask);
        else
          mma_commit(&empty[stage]);
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      };
      for (int u = unit0; u < num_units && ok && !*abort_flag; u += unit_step) {
        if constexpr (kChunked) {
          uint32_t d = 0;
          // kc: k-block index within the current accumulation chunk
          for (int kb = 0, kc = 0; kb < src.num_kb; ++kb) {
            if (kc == 0) {  // a chunk starts: take the next accumulator
              if (!mbar_wait(&tempty[acc], acc_phase ^ 1)) {
                ok = false;
                break;
              }
              tc_fence_after();
              d = tmem_base + uint32_t(acc * Cfg::ACC_STRIDE);
            }
            if (!mbar_wait(&full[stage], phase)) {
              ok = false;
              break;
            }
            tc_fence_after();
            mma_kblock(d, kc == 0);
            if (++kc == kb_chunk || kb == src.num_kb - 1) {  // the chunk (or the tile) is done
              kc = 0;
              mma_commit(&tfull[acc]);
              if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
              }
            }
          }
          if (!ok) break;
        } else {
          if (!mbar_wait(&tempty[acc], acc_phase ^ 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + uint32_t(acc * Cfg::ACC_STRIDE);
          for (int kb = 0; kb < src.num_kb; ++kb) {
            if (!mbar_wait(&full[stage], phase)) {
              ok = false;
              break;
            }
            tc_fence_after();
            mma_kblock(d, kb == 0);
          }
          if (!ok) break;
          mma_commit(&tfull[acc]);
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1;
          }
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
  } else if (warp >= 2 + kEpiWarps) {
    // ---------------------------------------------------------- converters
    if constexpr (kConv > 0) {
      const ConvCtx c{smem, Cfg::STAGE_BYTES, P * Cfg::A_BYTES, S, full, empty, abort_flag, status, scratch,
                      num_tiles};
      src.template convert<Op>(c);
    } else if constexpr (kLo != 0) {
      // lo planes: stage by stage, in the producer's order
      const int ct = int(threadIdx.x) - 32 * (2 + kEpiWarps);
      int stage = 0;
      uint32_t phase = 0;
      bool failed = false;
      for (int u = unit0; u < num_units && !failed; u += unit_step) {
        for (int kb = 0; kb < src.num_kb; ++kb) {
          bool ok = mbar_wait(&loaded[stage], phase);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok || __any_sync(0xffffffffu, *abort_flag)) {
            if (!ok) {
              record_error(status, GF_DEV_WAIT_TIMEOUT);
              *abort_flag = 1;
            }
            failed = true;
            break;
          }
          uint8_t* st = smem + stage * Cfg::STAGE_BYTES;
          if constexpr (kLo & 1) split_lo_tile<Cfg::A_BYTES>(st, st + Cfg::A_BYTES, ct);
          if constexpr (kLo & 2) split_lo_tile<Cfg::B_BYTES>(st + 2 * Cfg::A_BYTES, st + 2 * Cfg::A_BYTES + Cfg::B_BYTES, ct);
          fence_proxy_async_smem();  // the tensor core reads what these threads wrote
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    constexpr int H = epi_halves(BN), BNW = BN / H;
    const int quad = warp & 3;  // TMEM lanes this warp may read: 32*quad ..
    const int row = quad * 32 + lane;
    const int half = (warp - 2) >> 2;
    int acc = 0;
    uint32_t acc_phase = 0;
    // narrow tiles (H == 1): the second set of epilogue warps idles
    if constexpr (kChunked) {
      // running total of the tile's earlier chunks: TMEM columns
      // half * ACC_STRIDE + BN .. + BNW - 1 of this warp's lanes
      const int nchunks = (src.num_kb + kb_chunk - 1) / kb_chunk;
      const uint32_t tot = tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(half * Cfg::ACC_STRIDE + BN);
      bool failed = false;
      for (int u = unit0; half < H && u < num_units && !failed; u += unit_step) {
        const Tile tile = unit_tile(u);
        const Tile part{tile.b, tile.r0, tile.n0 + half * BNW, tile.nb * H + half};
        for (int c = 0; c < nchunks; ++c) {
          bool ok = mbar_wait(&tfull[acc], acc_phase);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok || __any_sync(0xffffffffu, *abort_flag)) {
            if (!ok) {
              record_error(status, GF_DEV_WAIT_TIMEOUT);
              *abort_flag = 1;
            }
            failed = true;
            break;
          }
          tc_fence_after();
          const uint32_t taddr =
              tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(acc * Cfg::ACC_STRIDE + half * BNW);
          if (c < nchunks - 1) {
#pragma unroll 1
            for (int j = 0; j < BNW; j += 16) {
              uint32_t r[16], q[16];
              GF_TMEM_LD16(taddr + uint32_t(j), r);
              if (c > 0) GF_TMEM_LD16(tot + uint32_t(j), q);
              GF_TMEM_WAIT16(r);
              if (c > 0) {
                GF_TMEM_WAIT16(q);
#pragma unroll
                for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(q[i]) + __uint_as_float(r[i]));
              }
              GF_TMEM_ST16(tot + uint32_t(j), r);
            }
            tmem_wait_st();  // the next chunk reads the total back
          } else {
            Epi::template apply_last<BNW>(ep, taddr, tot, part, row, c > 0);
          }
          tc_fence_before();
          mbar_arrive(&tempty[acc]);
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1;
          }
        }
      }
    } else {
      constexpr bool kTma = epi_tma_store<Epi, Op>();
      BoxStore st{};
      if constexpr (kTma) {
        st.buf = boxes + (warp - 2) * 2 * kStoreBoxFloats;
        st.map = &maps.c;
      }
      for (int u = unit0; half < H && u < num_units; u += unit_step) {
        const Tile tile = unit_tile(u);
        bool ok = mbar_wait(&tfull[acc], acc_phase);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok || __any_sync(0xffffffffu, *abort_flag)) {
          if (!ok) {
            record_error(status, GF_DEV_WAIT_TIMEOUT);
            *abort_flag = 1;
          }
          break;
        }
        tc_fence_after();
        const uint32_t taddr =
            tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(acc * Cfg::ACC_STRIDE + half * BNW);
        const Tile part{tile.b, tile.r0, tile.n0 + half * BNW, tile.nb * H + half};
        bool live = true;
        if constexpr (CL > 1) live = src.live(tile);  // not a tile wholly past M
        if (!live) {
        } else if constexpr (EpiTma<Epi>::value) {
          st.y = part.r0 + quad * 32;
          Epi::template apply<BNW, kTma>(ep, taddr, part, row, st);
        } else {
          Epi::template apply<BNW>(ep, taddr, part, row);
        }
        tc_fence_before();
        mbar_arrive(&tempty[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if constexpr (kTma) {  // the warp's boxes are written out before the CTA ends
        if (lane == 0) bulk_wait<0>();
        __syncwarp();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // (CL > 1) every copy into and arrival on this CTA's shared memory from the
  // other CTAs has landed (the producer's waits above): the cluster leaves
  // together
  if constexpr (CL > 1) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

// Host: launch the persistent kernel, one CTA per SM (or per unit of work
// when there are fewer), on the caller's stream, with the dominant-kernel
// profiling marks around it.  `units` = tiles, or (CL > 1) groups of CL
// tiles; the clusters go through cudaLaunchKernelEx, as many as can be
// resident at once.
template <int BN, class Op, class Src, class Epi, int CL = 1>
gf_status launch_gemm(const DeviceInfo& dev, const OperandMaps& maps, const Src& src, int64_t units,
                      const typename Epi::Params& ep, cudaStream_t stream) {
  using Cfg = TileCfg<BN, Op, SrcConv<Src>::scratch + epi_smem_bytes<Epi, Op>()>;
  auto kern = gemm_tc_kernel<BN, Op, Src, Epi, CL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
    return GF_ERR_CUDA;
  constexpr int threads = gemm_threads<Src, Epi, Op, BN>();
  if constexpr (CL == 1) {
    const int grid = int(units < dev.sm_count ? units : dev.sm_count);
    profile_mark_begin(stream);
    kern<<<grid, threads, Cfg::SMEM_BYTES, stream>>>(maps, src, ep, device_status_word());
    profile_mark_end(stream);
    return cudaGetLastError() == cudaSuccess ? GF_OK : GF_ERR_CUDA;
  } else {
    cudaLaunchConfig_t cfg{};
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(unsigned(CL * (dev.sm_count / CL)), 1, 1);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1) return GF_ERR_CUDA;
    const int64_t n = units < clusters ? units : clusters;
    cfg.gridDim = dim3(unsigned(CL * n), 1, 1);
    profile_mark_begin(stream);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, maps, src, ep, device_status_word());
    profile_mark_end(stream);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? GF_OK : GF_ERR_CUDA;
  }
}

}  // namespace gf
