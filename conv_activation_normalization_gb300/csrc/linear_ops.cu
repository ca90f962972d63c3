// The two Linear-based chains:
//   gf_linear_swish_bias_groupnorm   (page Kimi-K2.6__l2_p37)
//   gf_linear_lse_act                (page Kimi-K2.6__l2_p64)
// Both run a hi/lo split pre-pass on x and W, then one persistent tcgen05
// GEMM (3xTF32, BF16 or 3xBF16) whose epilogue does the rest of the chain
// on the accumulator tile in registers; the logsumexp chain adds a tiny
// per-row merge kernel, and GroupNorm groups other than 16-128 columns wide
// a per-row normalisation kernel.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <type_traits>

#include "gemm_tc.cuh"
#include "host_common.h"
#include "host_pipe.h"
#include "kernels_common.cuh"

namespace gf {

// ------------------------------------------------------------- epilogues
// Linear -> Swish -> +bias -> GroupNorm on a 128 x BN accumulator tile; one
// thread owns one row.  A group is gw consecutive columns (gw = 16, 32, 64 or
// 128).  Columns are handled 64 at a time: the mean and the (two-pass,
// biased) variance of each 16-column quarter's group are formed in the
// thread's registers.  A 128-column group spans two such halves: the first
// half's t is parked in TMEM (over its accumulator), the halves' (mean, M2)
// are merged with the pairwise update of Chan, Golub and LeVeque, and the
// first half is read back for its output.  The output goes out with plain
// stores, or (TMA) as boxes of 32 rows x 16 columns written to shared memory
// and sent by TMA stores.
struct GNParams {
  const float* b_lin;  // may be null
  const float* bias;
  const float* gamma;
  const float* beta;
  float* out;
  int M, N;
  float eps;
  int gw;              // group width (the epilogue's GW)
};
template <int GW>
struct EpiSwishBiasGNT {
  static_assert(GW == 16 || GW == 32 || GW == 64 || GW == 128, "group width");
  static constexpr bool kFixedBN = false;
  // narrowest tile whose epilogue warps own whole groups: a 128-column group
  // takes a warp's whole half of a 256-column tile
  static constexpr int kMinBN = GW == 128 ? 256 : 64;
  static constexpr int kTileGW = GW;  // the group width the tile-width rule sees
  static constexpr bool kTmaStore = true;  // the output may go out as TMA-stored boxes
  using Params = GNParams;

  // t = Swish(y + b_lin) + bias over the 64 columns n0.., in place; q[i] =
  // sum of quarter i's t.  Quarters from nq on lie past the last column
  // (N is a multiple of the group width, so only when GW < 64) and are left
  // alone.
  __device__ __forceinline__ static void swish_bias(const Params& p, int n0, int nq, float (&v)[64], float (&q)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      q[i] = 0.f;
      if (i >= nq) continue;  // uniform across the warp
      float2 sum = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 16 * i; j < 16 * i + 16; j += 4) {
        const float4 bl = p.b_lin ? __ldg(reinterpret_cast<const float4*>(p.b_lin + n0 + j)) : make_float4(0, 0, 0, 0);
        const float4 bb = __ldg(reinterpret_cast<const float4*>(p.bias + n0 + j));
        const float2 a = add2(swish2(add2(make_float2(v[j], v[j + 1]), make_float2(bl.x, bl.y))),
                              make_float2(bb.x, bb.y));
        const float2 c = add2(swish2(add2(make_float2(v[j + 2], v[j + 3]), make_float2(bl.z, bl.w))),
                              make_float2(bb.z, bb.w));
        v[j] = a.x;
        v[j + 1] = a.y;
        v[j + 2] = c.x;
        v[j + 3] = c.y;
        sum = add2(sum, add2(a, c));
      }
      q[i] = sum.x + sum.y;
    }
  }
  // per quarter: the sum of its group's quarters (GW <= 64)
  __device__ __forceinline__ static void group_sums(const float (&q)[4], float (&g)[4]) {
    const float s01 = q[0] + q[1], s23 = q[2] + q[3], s = s01 + s23;
    g[0] = GW == 16 ? q[0] : GW == 32 ? s01 : s;
    g[1] = GW == 16 ? q[1] : GW == 32 ? s01 : s;
    g[2] = GW == 16 ? q[2] : GW == 32 ? s23 : s;
    g[3] = GW == 16 ? q[3] : GW == 32 ? s23 : s;
  }
  // sum of squared deviations of quarter i's t from mu[i]
  __device__ __forceinline__ static void quarter_m2(const float (&v)[64], const float (&mu)[4], float (&m2)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 nm = make_float2(-mu[i], -mu[i]);
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 16 * i; j < 16 * i + 16; j += 2) {
        const float2 d = add2(make_float2(v[j], v[j + 1]), nm);
        acc = fma2(d, d, acc);
      }
      m2[i] = acc.x + acc.y;
    }
  }
  // (t - mu) rstd gamma + beta over the 64 columns n0.. of the row (the
  // first nq quarters)
  __device__ __forceinline__ static void normalize_store(const Params& p, int n0, int nq, const float (&v)[64],
                                                         const float (&mu)[4], const float (&rstd)[4], float* orow,
                                                         bool valid) {
#pragma unroll
    for (int j = 0; j < 64; j += 4) {
      if (j / 16 >= nq) break;  // uniform across the warp
      const float2 nm = make_float2(-mu[j / 16], -mu[j / 16]), r2 = make_float2(rstd[j / 16], rstd[j / 16]);
      const float4 ga = __ldg(reinterpret_cast<const float4*>(p.gamma + n0 + j));
      const float4 be = __ldg(reinterpret_cast<const float4*>(p.beta + n0 + j));
      const float2 a = fma2(mul2(add2(make_float2(v[j], v[j + 1]), nm), r2), make_float2(ga.x, ga.y),
                            make_float2(be.x, be.y));
      const float2 c = fma2(mul2(add2(make_float2(v[j + 2], v[j + 3]), nm), r2), make_float2(ga.z, ga.w),
                            make_float2(be.z, be.w));
      if (valid) __stcs(reinterpret_cast<float4*>(orow + j), make_float4(a.x, a.y, c.x, c.y));
    }
  }
  // The same values for quarter J0 / 16 (columns n0 + J0 ..  + 15), sent as
  // one box: lane l writes its row's 64 bytes into row l of a box with the
  // 64-byte swizzle (16-byte piece c of row l at piece c ^ ((l >> 1) & 3):
  // the warp's 16-byte writes hit distinct banks in each group of 8 lanes),
  // then lane 0 stores the box at output column n0 + J0, row st.y (rows past
  // M are not written).  The values are formed first; the buffer, used two
  // boxes earlier, is rewritten once that box's store has read it.
  template <int J0>
  __device__ __forceinline__ static void normalize_box(const Params& p, int n0, const float (&v)[64], float mu,
                                                       float rstd, BoxStore& st) {
    const int lane = int(threadIdx.x & 31);
    const float2 nm = make_float2(-mu, -mu), r2 = make_float2(rstd, rstd);
    float4 o[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int j = J0 + 4 * c;
      const float4 ga = __ldg(reinterpret_cast<const float4*>(p.gamma + n0 + j));
      const float4 be = __ldg(reinterpret_cast<const float4*>(p.beta + n0 + j));
      const float2 a = fma2(mul2(add2(make_float2(v[j], v[j + 1]), nm), r2), make_float2(ga.x, ga.y),
                            make_float2(be.x, be.y));
      const float2 d = fma2(mul2(add2(make_float2(v[j + 2], v[j + 3]), nm), r2), make_float2(ga.z, ga.w),
                            make_float2(be.z, be.w));
      o[c] = make_float4(a.x, a.y, d.x, d.y);
    }
    float* b = st.buf + (st.n & 1) * kStoreBoxFloats;
    if (st.n >= 2) {
      if (lane == 0) bulk_wait_read<1>();
      __syncwarp();
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) *reinterpret_cast<float4*>(b + lane * 16 + ((c ^ ((lane >> 1) & 3)) << 2)) = o[c];
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(st.map, smem_u32(b), n0 + J0, st.y);
      bulk_commit();
    }
    ++st.n;
  }
  // the normalised 64 columns n0.. (their first nq quarters) of the row:
  // boxes (TMA) or plain stores
  template <bool TMA>
  __device__ __forceinline__ static void emit(const Params& p, int n0, int nq, const float (&v)[64],
                                              const float (&mu)[4], const float (&rstd)[4], float* orow, bool valid,
                                              BoxStore& st) {
    if constexpr (TMA) {
      normalize_box<0>(p, n0, v, mu[0], rstd[0], st);
      if (nq > 1) normalize_box<16>(p, n0, v, mu[1], rstd[1], st);  // (nq uniform across the warp)
      if (nq > 2) normalize_box<32>(p, n0, v, mu[2], rstd[2], st);
      if (nq > 3) normalize_box<48>(p, n0, v, mu[3], rstd[3], st);
    } else {
      normalize_store(p, n0, nq, v, mu, rstd, orow, valid);
    }
  }

  template <int BN, bool TMA>
  __device__ __forceinline__ static void apply(const Params& p, uint32_t taddr, const Tile& t, int row,
                                               BoxStore& st) {
    const int m = t.r0 + row;
    const bool valid = m < p.M;
    float* orow = p.out + size_t(m) * size_t(p.N);
    if constexpr (GW == 128) {  // the warp's 128 columns are one group
      static_assert(GW != 128 || BN == 128, "128-column groups need 256-column tiles");
      const int n0 = t.n0;
      if (n0 >= p.N) return;  // uniform across the warp
      float v[64], q[4], mu[4], m2[4], rs[4];
      // first half: t and its (mean, M2); t parked over the accumulator
      tmem_load64(taddr, v);
      swish_bias(p, n0, 4, v, q);
      const float mean0 = (q[0] + q[1] + q[2] + q[3]) * (1.f / 64.f);
#pragma unroll
      for (int i = 0; i < 4; ++i) mu[i] = mean0;
      quarter_m2(v, mu, m2);
      const float m2a = m2[0] + m2[1] + m2[2] + m2[3];
      {
        uint32_t lo[32], hi[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          lo[i] = __float_as_uint(v[i]);
          hi[i] = __float_as_uint(v[32 + i]);
        }
        GF_TMEM_ST32(taddr, lo);
        GF_TMEM_ST32(taddr + 32, hi);
      }
      // second half
      tmem_load64(taddr + 64, v);
      swish_bias(p, n0 + 64, 4, v, q);
      const float mean1 = (q[0] + q[1] + q[2] + q[3]) * (1.f / 64.f);
#pragma unroll
      for (int i = 0; i < 4; ++i) mu[i] = mean1;
      quarter_m2(v, mu, m2);
      const float m2b = m2[0] + m2[1] + m2[2] + m2[3];
      // merge the halves: M2 = M2a + M2b + delta^2 * 64 * 64 / 128
      const float delta = mean1 - mean0;
      const float mean = 0.5f * (mean0 + mean1);
      const float rstd = rsqrtf((m2a + m2b + delta * delta * 32.f) * (1.f / 128.f) + p.eps);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        mu[i] = mean;
        rs[i] = rstd;
      }
      emit<TMA>(p, n0 + 64, 4, v, mu, rs, orow + n0 + 64, valid, st);
      tmem_wait_st();
      tmem_load64(taddr, v);
      emit<TMA>(p, n0, 4, v, mu, rs, orow + n0, valid, st);
    } else {
#pragma unroll 1
      for (int g = 0; g < BN / 64; ++g) {
        const int n0 = t.n0 + g * 64;
        if (n0 >= p.N) break;  // uniform across the warp
        // quarters inside the row (all four unless GW < 64 and N % 64 != 0)
        const int nq = GW >= 64 ? 4 : min(4, (p.N - n0) / 16);
        float v[64], q[4], mu[4], m2[4], rs[4];
        tmem_load64(taddr + uint32_t(g * 64), v);
        swish_bias(p, n0, nq, v, q);
        if constexpr (GW == 64) {  // one group: one mean, one M2
          float2 sum = make_float2(0.f, 0.f);
#pragma unroll
          for (int i = 0; i < 4; ++i) sum.x += q[i];
          const float mean = sum.x * (1.f / 64.f);
          const float2 nmean = make_float2(-mean, -mean);
          float2 acc = make_float2(0.f, 0.f);
#pragma unroll
          for (int j = 0; j < 64; j += 2) {
            const float2 d = add2(make_float2(v[j], v[j + 1]), nmean);
            acc = fma2(d, d, acc);
          }
          const float rstd = rsqrtf((acc.x + acc.y) * (1.f / 64.f) + p.eps);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            mu[i] = mean;
            rs[i] = rstd;
          }
          emit<TMA>(p, n0, nq, v, mu, rs, orow + n0, valid, st);
        } else {
          constexpr float inv = 1.f / float(GW);  // a power of two: exact
          float gs[4], gm2[4];
          group_sums(q, gs);
#pragma unroll
          for (int i = 0; i < 4; ++i) mu[i] = gs[i] * inv;
          quarter_m2(v, mu, m2);
          group_sums(m2, gm2);
#pragma unroll
          for (int i = 0; i < 4; ++i) rs[i] = rsqrtf(gm2[i] * inv + p.eps);
          emit<TMA>(p, n0, nq, v, mu, rs, orow + n0, valid, st);
        }
      }
    }
  }
};

// Any other group width: the epilogue stores t = Swish(y + b_lin) + bias
// and gn_rows_kernel normalises the rows in place afterwards (one more pass
// over the output, instead of none).
struct EpiSwishBiasStore {
  static constexpr bool kFixedBN = false;
  static constexpr int kMinBN = 64;
  static constexpr int kTileGW = 0;
  using Params = GNParams;
  template <int BN>
  __device__ __forceinline__ static void apply(const Params& p, uint32_t taddr, const Tile& t, int row) {
    const int m = t.r0 + row;
    const bool valid = m < p.M;
    float* orow = p.out + size_t(m) * size_t(p.N);
#pragma unroll 1
    for (int g = 0; g < BN / 32; ++g) {
      const int n0 = t.n0 + g * 32;
      if (n0 >= p.N) break;  // uniform across the warp
      uint32_t v[32];
      GF_TMEM_LD32(taddr + uint32_t(g * 32), v);
      GF_TMEM_WAIT32(v);
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const int n = n0 + j;
        const bool in0 = n < p.N, in1 = n + 1 < p.N;
        const float b0 = p.b_lin && in0 ? __ldg(p.b_lin + n) : 0.f, b1 = p.b_lin && in1 ? __ldg(p.b_lin + n + 1) : 0.f;
        const float2 sv = swish2(make_float2(__uint_as_float(v[j]) + b0, __uint_as_float(v[j + 1]) + b1));
        if (valid && in0) orow[n] = sv.x + __ldg(p.bias + n);
        if (valid && in1) orow[n + 1] = sv.y + __ldg(p.bias + n + 1);
      }
    }
  }
};

// GroupNorm of each row of out[M][N] in place, groups of gw consecutive
// columns: one block per row, one warp per group at a time, the group's
// mean and centred second moment in two passes (fp32, lane-strided sums and
// a shuffle tree), then (t - mean) rstd gamma + beta.
__global__ void __launch_bounds__(256) gn_rows_kernel(float* __restrict__ out, const float* __restrict__ gamma,
                                                      const float* __restrict__ beta, int N, int gw, float eps) {
  float* row = out + size_t(blockIdx.x) * N;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const float inv = 1.f / float(gw);
  for (int g = warp; g < N / gw; g += 8) {
    float* v = row + size_t(g) * gw;
    float s = 0.f;
    for (int i = lane; i < gw; i += 32) s += v[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float mean = s * inv;
    float q = 0.f;
    for (int i = lane; i < gw; i += 32) {
      const float d = v[i] - mean;
      q = fmaf(d, d, q);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
    const float rstd = rsqrtf(q * inv + eps);
    for (int i = lane; i < gw; i += 32) {
      const int n = g * gw + i;
      v[i] = fmaf((v[i] - mean) * rstd, __ldg(gamma + n), __ldg(beta + n));
    }
  }
}

// Runs f(TypeTag<epilogue>) with the fused epilogue of group width ep.gw
// (16, 32, 64 or 128 columns), or with EpiSwishBiasStore followed by
// gn_rows_kernel on stream s for any other width.
template <class T>
struct TypeTag {
  using type = T;
};
template <class F>
gf_status with_gn_epilogue(const GNParams& ep, cudaStream_t s, F&& f) {
  switch (ep.gw) {
    case 16: return f(TypeTag<EpiSwishBiasGNT<16>>{});
    case 32: return f(TypeTag<EpiSwishBiasGNT<32>>{});
    case 64: return f(TypeTag<EpiSwishBiasGNT<64>>{});
    case 128: return f(TypeTag<EpiSwishBiasGNT<128>>{});
    default: {
      const gf_status st = f(TypeTag<EpiSwishBiasStore>{});
      if (st != GF_OK) return st;
      gn_rows_kernel<<<unsigned(ep.M), 256, 0, s>>>(ep.out, ep.gamma, ep.beta, ep.N, ep.gw, ep.eps);
      return cuda_status(cudaGetLastError());
    }
  }
}

// Linear -> per-row (max, sum exp(y - max)) over the tile's columns, written
// as one float2 partial per (row, epilogue column half); columns are read 16
// at a time and merged online, so BN may be any multiple of 16 (the tile
// widths are 160, 224 and 256).
//
// The chain's K is long (8192 in the pages' problem), so in the
// three-product modes the accumulator is taken in chunks of kChunkK
// (chunked(), see gemm_tc.cuh): the kernel keeps the running total of the
// earlier chunks in spare TMEM columns and hands it to apply_last with the
// last chunk.  The one-product BF16 mode (3e-2 tolerance) reads its single
// chunk with apply.
struct EpiLSEPartial {
  static constexpr bool kFixedBN = true;  // the partials' layout follows the tile width
  static constexpr int kChunkK = 1024;    // K elements per accumulation chunk
  template <class Op>
  __host__ __device__ static constexpr bool chunked() {
    return Op::kProducts == 3;
  }
  struct Params {
    const float* b;  // may be null
    float2* part;    // [M][n_blocks]: one per row and epilogue column range
    int M, N, n_blocks;
  };
  // v[j] (+ bias, -inf past N) of one 16-column piece folded into (mx, s)
  __device__ __forceinline__ static void merge_piece(const Params& p, int n0, float (&v)[16], float& mx, float& s) {
    float cm = -INFINITY;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int n = n0 + j;
      const float bj = (p.b && n < p.N) ? __ldg(p.b + n) : 0.f;
      v[j] = n < p.N ? v[j] + bj : -INFINITY;
      cm = fmaxf(cm, v[j]);
    }
    const float nm = fmaxf(mx, cm);
    s *= __expf(mx - nm);
#pragma unroll
    for (int j = 0; j < 16; ++j) s += __expf(v[j] - nm);
    mx = nm;
  }
  template <int BN>
  __device__ __forceinline__ static void apply(const Params& p, uint32_t taddr, const Tile& t, int row) {
    static_assert(BN % 16 == 0, "16-column pieces");
    const int m = t.r0 + row;
    float mx = -INFINITY, s = 0.f;
#pragma unroll 1
    for (int g = 0; g < BN / 16; ++g) {
      const int n0 = t.n0 + g * 16;
      if (n0 >= p.N) break;  // uniform across the warp
      uint32_t r[16];
      GF_TMEM_LD16(taddr + uint32_t(g * 16), r);
      GF_TMEM_WAIT16(r);
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
      merge_piece(p, n0, v, mx, s);
    }
    if (m < p.M) p.part[size_t(m) * p.n_blocks + t.nb] = make_float2(mx, s);
  }
  // the last chunk at taddr plus, when `earlier`, the earlier chunks' total
  // at tot (both TMEM addresses of the thread's lane)
  template <int BN>
  __device__ __forceinline__ static void apply_last(const Params& p, uint32_t taddr, uint32_t tot, const Tile& t,
                                                    int row, bool earlier) {
    const int m = t.r0 + row;
    float mx = -INFINITY, s = 0.f;
#pragma unroll 1
    for (int g = 0; g < BN / 16; ++g) {
      const int n0 = t.n0 + g * 16;
      if (n0 >= p.N) break;  // uniform across the warp
      uint32_t r[16], q[16];
      GF_TMEM_LD16(taddr + uint32_t(g * 16), r);
      if (earlier) GF_TMEM_LD16(tot + uint32_t(g * 16), q);
      GF_TMEM_WAIT16(r);
      float v[16];
      if (earlier) {
        GF_TMEM_WAIT16(q);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(q[j]) + __uint_as_float(r[j]);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
      }
      merge_piece(p, n0, v, mx, s);
    }
    if (m < p.M) p.part[size_t(m) * p.n_blocks + t.nb] = make_float2(mx, s);
  }
};

// Plain Linear: out[m, n] = acc + b[n] (the contraction step alone).
struct EpiStore {
  static constexpr bool kFixedBN = false;
  struct Params {
    const float* b;  // may be null
    float* out;
    int M, N;
  };
  static constexpr int kMinBN = 64;
  static constexpr int kTileGW = 0;
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
    if (q.x == -INFINITY) continue;  // a column range with no valid column
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

// 3xTF32 operands whose lo plane the GEMM computes in the SM from the raw
// fp32 tile (bit 0: x, bit 1: W) instead of reading a plane a pre-pass wrote
// (gemm_tc_kernel, kLoInSm): the GroupNorm chain at 64-column tiles, where
// few rows leave the GEMM waiting on operand bytes and the pre-passes are a
// large part of the call (M = 256: 42.0 -> 30.9 us per call, M = 512:
// 60.1 -> 51.1; level at 128 columns).  Where the MMAs bound the GEMM, the
// conversion's shared-memory traffic slows them more than the pre-pass costs
// (M = 32768: 0.972 -> 1.204 ms), and the same held for the Conv1d's weights.
// The logsumexp chain takes W's lo plane in the SM (bit 1): its W (8192 x
// 8192, 268 MB) streams from DRAM, so the pre-pass's read and write of it
// cost more than the GEMM loses to the conversion (step 0.5775 -> 0.5682 ms
// on x[1024,8192]; outputs bit-identical).
template <class Epi>
constexpr int lo_mask_at(int mode, int bn) {
  constexpr bool gn = !std::is_same<Epi, EpiLSEPartial>::value && !std::is_same<Epi, EpiStore>::value;
  if constexpr (std::is_same<Epi, EpiLSEPartial>::value) return mode == GF_MODE_FP32_3XTF32 ? 2 : 0;
  return gn && mode == GF_MODE_FP32_3XTF32 && bn == 64 ? 3 : 0;
}
// CTAs per cluster of the BF16 GroupNorm kernel at 256 columns: two take
// 0.2071 ms at M = 32768 against 0.2103 for one; four time the same as two.
constexpr int kClusterBF16 = 2;

// Tile width of the LSE chain.  In the three-product modes 160 columns: the
// tile fits three smem stages (two for 224 or 256), deep enough for the
// mainloop to keep pace with W streaming from DRAM (1024 x 8192 x 8192: 95 %
// of the 3xTF32 peak against 82 % with 224-column tiles and two stages), and
// its chunked accumulation finds room for the running totals in TMEM.
// The one-product BF16 mode has four or more stages at any width and no
// chunking; there 224 or 256 columns, whichever gives fewer waves x per-tile
// time.
constexpr int kLseWidths[3] = {160, 224, 256};
int lse_tile_width(int64_t M, int64_t N, int sm_count, int32_t mode) {
  if (mode != GF_MODE_BF16) return 160;
  const int64_t mb = (M + 127) / 128;
  int best = 224;
  double best_t = 0.0;
  for (int bn : {224, 256}) {
    const int64_t tiles = mb * ((N + bn - 1) / bn);
    const int64_t waves = (tiles + sm_count - 1) / sm_count;
    const double t = double(waves) * bn;
    if (best_t == 0.0 || t < best_t) {
      best = bn;
      best_t = t;
    }
  }
  return best;
}
// Partials per row for a tile width: one per epilogue column half.
int64_t lse_parts(int64_t N, int bn) { return (N + bn - 1) / bn * epi_halves(bn); }

// The GEMM tile width (columns per CTA tile) of a call: for the logsumexp
// chain the width lse_tile_width picks; otherwise 256 columns when that gives
// every SM at least one tile, else 128 or 64 (small M), trading per-tile
// efficiency for parallelism; a fused 128-column GroupNorm group (gw = 128)
// always takes 256-column tiles (a warp's half-tile is one group).  gw is the
// fused epilogue's group width, 0 for the other epilogues.  The dispatch and
// gf_linear_tile_width both use this function.
int linear_tile_width(bool lse, int64_t M, int64_t N, int gw, int32_t mode, int sm_count) {
  if (lse) return lse_tile_width(M, N, sm_count, mode);
  if (gw == 128) return 256;
  const int64_t mb = (M + kBM - 1) / kBM;
  if (mb * ((N + 255) / 256) >= sm_count) return 256;
  if (mb * ((N + 127) / 128) >= sm_count) return 128;
  return 64;
}

// Group widths the GEMM epilogue normalises itself (others: gn_rows_kernel).
bool gn_fused_width(int64_t gw) { return gw == 16 || gw == 32 || gw == 64 || gw == 128; }

bool mode_ok(int32_t mode) {
  return mode == GF_MODE_FP32_3XTF32 || mode == GF_MODE_BF16 || mode == GF_MODE_FP32_3XBF16;
}

// Bytes of one operand's pre-pass planes in the workspace: the lo plane
// (3xTF32: hi is the raw tensor), bf16 hi (BF16) or bf16 hi + lo (3xBF16).
// K padded to a whole number of 16-byte rows (4 fp32, 8 bf16 elements) for
// the TMA: the pre-pass then writes every plane of the operand, zeros in
// the padding columns.
int64_t kpad(int64_t K, int32_t mode) {
  const int64_t q = mode == GF_MODE_FP32_3XTF32 ? 4 : 8;
  return (K + q - 1) / q * q;
}

size_t operand_ws_bytes(int64_t rows, int64_t K, int32_t mode) {
  const int64_t Kp = kpad(K, mode);
  if (Kp != K) {  // padded planes: fp32 hi + lo, bf16 hi, or bf16 hi + lo
    const size_t n = size_t(rows) * size_t(Kp);
    return align_up(n * (mode == GF_MODE_FP32_3XTF32 ? 8 : mode == GF_MODE_BF16 ? 2 : 4), 256);
  }
  const size_t n = size_t(rows) * size_t(K);
  switch (mode) {
    case GF_MODE_FP32_3XTF32: return align_up(n * 4, 256);
    case GF_MODE_BF16: return align_up(n * 2, 256);
    default: return align_up(n * 4, 256);  // two bf16 planes
  }
}

// M = 0 (an empty batch) passes: the entry points then return GF_OK
// without launching anything.
gf_status check_linear_shape(int64_t M, int64_t K, int64_t N, int32_t mode) {
  if (M < 0 || K < 1 || N < 1) return GF_ERR_SHAPE;
  // (a K that is not a whole number of 16-byte rows is padded by the
  // pre-pass: kpad)
  (void)mode;
  if (M > (int64_t(1) << 31) - 256 || N > (int64_t(1) << 31) - 256 || K > (int64_t(1) << 31) - 64)
    return GF_ERR_SHAPE;  // TMA coordinates are int32
  return GF_OK;
}

// GroupNorm groups: any count that divides N (groups of 16, 32, 64 or 128
// columns run in the GEMM epilogue, other widths in a second kernel).
bool gn_groups_ok(int64_t N, int32_t groups) { return groups >= 1 && N % groups == 0; }

// Planes the GEMM reads for one operand: p[0] = hi (or the only operand),
// p[1] = lo.
struct Planes {
  const void* p[2];
};

// Every plane of an operand whose rows are K wide, written with rows Kp
// wide (zeros in columns K .. Kp - 1): fp32 hi (the raw value) and lo in the
// 3xTF32 mode, bf16 hi (and lo) in the BF16 modes.
template <int MODE>
__global__ void split_padded_kernel(const float* __restrict__ src, int64_t rows, int K, int Kp, void* planes) {
  const size_t n = size_t(rows) * size_t(Kp);
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += size_t(gridDim.x) * blockDim.x) {
    const size_t r = i / size_t(Kp);
    const int k = int(i - r * size_t(Kp));
    const float v = k < K ? __ldg(src + r * size_t(K) + size_t(k)) : 0.f;
    if constexpr (MODE == GF_MODE_FP32_3XTF32) {
      float* p = static_cast<float*>(planes);
      p[i] = v;
      p[n + i] = v - tf32_hi(v);
    } else {
      __nv_bfloat16* p = static_cast<__nv_bfloat16*>(planes);
      const __nv_bfloat16 h = __float2bfloat16_rn(v);
      p[i] = h;
      if constexpr (MODE == GF_MODE_FP32_3XBF16) p[n + i] = __float2bfloat16_rn(v - __bfloat162float(h));
    }
  }
}

// Run the split pre-pass of one operand into `ws` and return its planes
// (rows kpad(K, mode) wide).
gf_status prepare_operand(const float* src, int64_t rows, int64_t K, int32_t mode, void* ws, const DeviceInfo& dev,
                          cudaStream_t s, Planes* out, bool need_lo = true) {
  const int64_t Kp = kpad(K, mode);
  if (Kp != K) {
    const size_t n = size_t(rows) * size_t(Kp);
    const size_t esz = mode == GF_MODE_FP32_3XTF32 ? 4 : 2;
    out->p[0] = ws;
    out->p[1] = mode == GF_MODE_BF16 ? nullptr : static_cast<uint8_t*>(ws) + n * esz;
    const int blocks = split_blocks((n + 3) / 4, dev.sm_count);
    switch (mode) {
      case GF_MODE_FP32_3XTF32:
        split_padded_kernel<GF_MODE_FP32_3XTF32><<<blocks, 256, 0, s>>>(src, rows, int(K), int(Kp), ws);
        break;
      case GF_MODE_BF16:
        split_padded_kernel<GF_MODE_BF16><<<blocks, 256, 0, s>>>(src, rows, int(K), int(Kp), ws);
        break;
      default:
        split_padded_kernel<GF_MODE_FP32_3XBF16><<<blocks, 256, 0, s>>>(src, rows, int(K), int(Kp), ws);
    }
    return cuda_status(cudaGetLastError());
  }
  const size_t n = size_t(rows) * size_t(K);
  switch (mode) {
    case GF_MODE_FP32_3XTF32:
      out->p[0] = src;
      out->p[1] = need_lo ? ws : nullptr;  // (else the GEMM computes lo itself)
      return need_lo ? launch_split_lo_tf32(src, static_cast<float*>(ws), n, dev.sm_count, s) : GF_OK;
    case GF_MODE_BF16:
      out->p[0] = ws;
      out->p[1] = nullptr;
      return launch_split_bf16(src, ws, nullptr, n, dev.sm_count, s);
    default: {
      void* lo = static_cast<uint8_t*>(ws) + n * 2;
      out->p[0] = ws;
      out->p[1] = lo;
      return launch_split_bf16(src, ws, lo, n, dev.sm_count, s);
    }
  }
}

template <int BN, class Op, class Epi>
gf_status run_linear_gemm(const DeviceInfo& dev, const Planes& a, const Planes& b, int64_t M, int64_t K, int64_t N,
                          int m_fastest, const typename Epi::Params& ep, cudaStream_t stream) {
  // The BF16 GroupNorm kernel at 256 columns runs in clusters of
  // kClusterBF16 CTAs that share each B tile (each CTA loads a slice of it):
  // its k-loop waits on operand bytes from L2 rather than on its MMAs.
  constexpr int CL = epi_tma_store<Epi, Op>() && BN == 256 ? kClusterBF16 : 1;
  constexpr int LO = lo_mask_at<Epi>(std::is_same<Op, OpTF32x3>::value ? GF_MODE_FP32_3XTF32 : GF_MODE_BF16, BN);
  using Src = LinearSrcT<LO>;
  OperandMaps maps{};
  const uint64_t da[2] = {uint64_t(K), uint64_t(M)};
  const uint32_t ba[2] = {uint32_t(Op::kBK), uint32_t(kBM)};
  const uint64_t db[2] = {uint64_t(K), uint64_t(N)};
  const uint32_t bb[2] = {uint32_t(Op::kBK), uint32_t(BN / CL)};
  for (int p = 0; p < Op::kPlanes; ++p) {
    gf_status st = GF_OK;
    if (p == 0 || !(LO & 1)) st = make_tmap(&maps.a[p], a.p[p], Op::kElem, 2, da, ba);
    if (st != GF_OK) return st;
    if (p == 0 || !(LO & 2)) st = make_tmap(&maps.b[p], b.p[p], Op::kElem, 2, db, bb);
    if (st != GF_OK) return st;
  }
  if constexpr (epi_tma_store<Epi, Op>()) {  // the output, in the epilogue's boxes of 32 rows x 16 columns
    const uint64_t dc[2] = {uint64_t(N), uint64_t(M)};
    const uint32_t bc[2] = {16u, 32u};
    const gf_status st = make_tmap(&maps.c, ep.out, 4, 2, dc, bc, 64);
    if (st != GF_OK) return st;
  }
  Src src;
  src.num_mb = int((M + kBM - 1) / kBM);
  src.num_nb = int((N + BN - 1) / BN);
  src.num_kb = int((K + Op::kBK - 1) / Op::kBK);
  if constexpr (epi_chunked<Epi, Op, BN>())
    src.kb_chunk = Epi::kChunkK / Op::kBK;  // (kChunkK is a multiple of kBK in every mode)
  else
    src.kb_chunk = src.num_kb;
  src.bn = BN;
  src.bk = Op::kBK;
  src.m_fastest = m_fastest;
  const int64_t units = int64_t(src.num_mb + CL - 1) / CL * src.num_nb;
  return launch_gemm<BN, Op, Src, Epi, CL>(dev, maps, src, units, ep, stream);
}

// The tile width the GEMM of epilogue Epi runs at: linear_tile_width's
// choice; a fused epilogue's groups must not straddle warps (Epi::kMinBN).
template <class Epi>
int gemm_tile_width(int64_t M, int64_t N, int32_t mode, int sm_count) {
  if constexpr (Epi::kFixedBN) {
    const int w = linear_tile_width(true, M, N, 0, mode, sm_count);
    return w == 160 || w == 224 ? w : kBNLinear;
  } else if constexpr (Epi::kMinBN > 128) {
    return 256;
  } else {
    const int w = linear_tile_width(false, M, N, Epi::kTileGW, mode, sm_count);
    return w == 256 || w == 128 ? w : 64;
  }
}

// Runs the GEMM at the tile width gemm_tile_width picks.  The LSE partials'
// layout follows the tile width (the caller sized them with the same
// function).
template <class Op, class Epi>
gf_status run_linear_gemm_bn(const DeviceInfo& dev, const Planes& a, const Planes& b, int64_t M, int64_t K,
                             int64_t N, int m_fastest, const typename Epi::Params& ep, cudaStream_t stream) {
  const int32_t mode = Op::kProducts == 1 ? GF_MODE_BF16 : GF_MODE_FP32_3XTF32;  // (only BF16 or not matters)
  if constexpr (Epi::kFixedBN) {
    switch (gemm_tile_width<Epi>(M, N, mode, dev.sm_count)) {
      case 160: return run_linear_gemm<160, Op, Epi>(dev, a, b, M, K, N, m_fastest, ep, stream);
      case 224: return run_linear_gemm<224, Op, Epi>(dev, a, b, M, K, N, m_fastest, ep, stream);
      default: return run_linear_gemm<kBNLinear, Op, Epi>(dev, a, b, M, K, N, m_fastest, ep, stream);
    }
  } else if constexpr (Epi::kMinBN > 128) {
    return run_linear_gemm<256, Op, Epi>(dev, a, b, M, K, N, m_fastest, ep, stream);
  } else {
    switch (gemm_tile_width<Epi>(M, N, mode, dev.sm_count)) {
      case 256: return run_linear_gemm<256, Op, Epi>(dev, a, b, M, K, N, m_fastest, ep, stream);
      case 128: return run_linear_gemm<128, Op, Epi>(dev, a, b, M, K, N, m_fastest, ep, stream);
      default: return run_linear_gemm<64, Op, Epi>(dev, a, b, M, K, N, m_fastest, ep, stream);
    }
  }
}

template <class Epi>
gf_status run_linear(int32_t mode, const DeviceInfo& dev, const Planes& a, const Planes& b, int64_t M, int64_t K,
                     int64_t N, int m_fastest, const typename Epi::Params& ep, cudaStream_t stream) {
  switch (mode) {
    case GF_MODE_FP32_3XTF32: return run_linear_gemm_bn<OpTF32x3, Epi>(dev, a, b, M, K, N, m_fastest, ep, stream);
    case GF_MODE_BF16: return run_linear_gemm_bn<OpBF16x1, Epi>(dev, a, b, M, K, N, m_fastest, ep, stream);
    default: return run_linear_gemm_bn<OpBF16x3, Epi>(dev, a, b, M, K, N, m_fastest, ep, stream);
  }
}

// Split both operands into the workspace, then run the fused GEMM.
template <class Epi>
gf_status split_and_run(int32_t mode, const float* x, const float* W, int64_t M, int64_t K, int64_t N, void* ws,
                        int m_fastest, const typename Epi::Params& ep, cudaStream_t s) {
  DeviceInfo dev;
  gf_status st = current_device(&dev);
  if (st != GF_OK) return st;
  Planes a, b;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  // (operands whose lo plane the GEMM computes itself need no split)
  const int lo = lo_mask_at<Epi>(mode, gemm_tile_width<Epi>(M, N, mode, dev.sm_count));
  if ((st = prepare_operand(x, M, K, mode, w8, dev, s, &a, !(lo & 1))) != GF_OK) return st;
  if ((st = prepare_operand(W, N, K, mode, w8 + operand_ws_bytes(M, K, mode), dev, s, &b, !(lo & 2))) != GF_OK)
    return st;
  return run_linear<Epi>(mode, dev, a, b, M, kpad(K, mode), N, m_fastest, ep, s);
}

}  // namespace
}  // namespace gf

using namespace gf;

extern "C" {

int32_t gf_linear_tile_width(int32_t chain, int64_t M, int64_t N, int32_t groups, int32_t mode, int32_t sm_count) {
  if (!mode_ok(mode) || sm_count < 1 || M < 0 || N < 1) return 0;
  switch (chain) {
    case GF_CHAIN_GROUPNORM: {
      if (!gn_groups_ok(N, groups)) return 0;
      const int64_t gw = N / groups;
      return linear_tile_width(false, M, N, gn_fused_width(gw) ? int(gw) : 0, mode, sm_count);
    }
    case GF_CHAIN_LSE: return linear_tile_width(true, M, N, 0, mode, sm_count);
    case GF_CHAIN_LINEAR: return linear_tile_width(false, M, N, 0, mode, sm_count);
    default: return 0;
  }
}

size_t gf_linear_swish_bias_groupnorm_workspace_size(int64_t M, int64_t K, int64_t N, int32_t groups,
                                                     int32_t mode) {
  if (!mode_ok(mode) || check_linear_shape(M, K, N, mode) != GF_OK || !gn_groups_ok(N, groups) || M == 0) return 0;
  return operand_ws_bytes(M, K, mode) + operand_ws_bytes(N, K, mode);
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
  // (an empty batch, M = 0, may pass NULL for x_planes and out)
  if ((M && (!x_planes || !out)) || !W_planes || !bias || !gamma || !beta) return GF_ERR_NULL;
  gf_status st = check_linear_shape(M, K, N, GF_MODE_FP32_3XTF32);
  if (st != GF_OK) return st;
  if (K % 4) return GF_ERR_SHAPE;  // the caller's planes are read with K-wide rows
  if (!gn_groups_ok(N, groups)) return GF_ERR_SHAPE;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return GF_ERR_SHAPE;
  if (!aligned16(x_planes) || !aligned16(W_planes) || !aligned16(bias) || !aligned16(gamma) || !aligned16(beta) ||
      !aligned16(out) || (b_lin && !aligned16(b_lin)))
    return GF_ERR_ALIGN;
  if (M == 0) return GF_OK;
  const Span ins[] = {{x_planes, size_t(M) * K * 8}, {W_planes, size_t(N) * K * 8}, {b_lin, size_t(N) * 4},
                      {bias, size_t(N) * 4},         {gamma, size_t(N) * 4},         {beta, size_t(N) * 4}};
  st = check_no_alias(Span{out, size_t(M) * N * 4}, ins, 6);
  if (st != GF_OK) return st;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != GF_OK) return st;
  const Planes a{{x_planes, x_planes + size_t(M) * K}}, b{{W_planes, W_planes + size_t(N) * K}};
  const GNParams ep{b_lin, bias, gamma, beta, out, int(M), int(N), eps, int(N / groups)};
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  return with_gn_epilogue(ep, s, [&](auto tag) {
    return run_linear<typename decltype(tag)::type>(GF_MODE_FP32_3XTF32, dev, a, b, M, K, N, 0, ep, s);
  });
}

gf_status gf_linear_swish_bias_groupnorm(const float* x, const float* W, const float* b_lin, const float* bias,
                                         const float* gamma, const float* beta, float* out, int64_t M,
                                         int64_t K, int64_t N, int32_t groups, float eps, int32_t mode,
                                         void* workspace, size_t workspace_bytes, void* stream) {
  if ((M && (!x || !out)) || !W || !bias || !gamma || !beta) return GF_ERR_NULL;
  if (!mode_ok(mode)) return GF_ERR_MODE;
  gf_status st = check_linear_shape(M, K, N, mode);
  if (st != GF_OK) return st;
  if (!gn_groups_ok(N, groups)) return GF_ERR_SHAPE;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return GF_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(W) || !aligned16(bias) || !aligned16(gamma) || !aligned16(beta) ||
      !aligned16(out) || (b_lin && !aligned16(b_lin)) || !aligned16(workspace))
    return GF_ERR_ALIGN;
  if (M == 0) return GF_OK;  // an empty batch: nothing to compute
  const size_t need = gf_linear_swish_bias_groupnorm_workspace_size(M, K, N, groups, mode);
  if (!workspace) return GF_ERR_NULL;
  if (workspace_bytes < need) return GF_ERR_WORKSPACE;
  const Span ins[] = {{x, size_t(M) * K * 4}, {W, size_t(N) * K * 4}, {b_lin, size_t(N) * 4},
                      {bias, size_t(N) * 4},  {gamma, size_t(N) * 4}, {beta, size_t(N) * 4},
                      {workspace, need}};
  st = check_no_alias(Span{out, size_t(M) * N * 4}, ins, 7);
  if (st != GF_OK) return st;
  const GNParams ep{b_lin, bias, gamma, beta, out, int(M), int(N), eps, int(N / groups)};
  // n-blocks fastest (m_fastest 0): the CTAs in flight share a few m-blocks
  // of x, while all of W stays resident in L2.
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  return with_gn_epilogue(ep, s, [&](auto tag) {
    return split_and_run<typename decltype(tag)::type>(mode, x, W, M, K, N, workspace, 0, ep, s);
  });
}

// ---------------------------------------------------------------- host path
namespace {

// Default rows per chunk: a whole number of waves of 128 x 256 tiles (the
// m-blocks per chunk times the n-blocks is a multiple of the SM count), at
// least 2048 rows: small enough that the pipeline's first copy-in and last
// copy-out are short, large enough to keep the per-chunk overheads small
// (32768 x 4096 output on 152 SMs: 2432-row chunks, 3.03 ms per call against
// 3.17 ms with 4864-row chunks, the copies being the bound).
int64_t host_chunk_rows(int64_t M, int64_t N, int sm_count) {
  const int64_t nb = (N + kBNLinear - 1) / kBNLinear;
  int64_t a = sm_count, b = nb;
  while (b) {
    const int64_t t = a % b;
    a = b;
    b = t;
  }
  const int64_t wave_mb = sm_count / a;  // m-blocks that fill whole waves
  int64_t mb = wave_mb;
  while (mb * kBM < 2048) mb += wave_mb;
  const int64_t rows = mb * kBM;
  return rows < M ? rows : M;
}

struct HostWs {
  size_t w_planes, x[2], xp[2], out[2], total;
};

HostWs host_ws(int64_t chunk, int64_t K, int64_t N, int32_t mode) {
  HostWs w{};
  size_t off = 0;
  w.w_planes = off;
  off += operand_ws_bytes(N, K, mode);
  for (int i = 0; i < 2; ++i) {
    w.x[i] = off;
    off += align_up(size_t(chunk) * K * 4, 256);
    w.xp[i] = off;
    off += operand_ws_bytes(chunk, K, mode);
    w.out[i] = off;
    off += align_up(size_t(chunk) * N * 4, 256);
  }
  w.total = off;
  return w;
}

// The CUDA side of gf_linear_swish_bias_groupnorm_host: chunks of rows of x
// in, rows of out back (the schedule and its streams: host_pipe.h).
struct CudaHostPipe final : CudaPipeBase {
  // inputs of the call
  const float* x_host;
  float* out_host;
  const float *W, *b_lin, *bias, *gamma, *beta;
  int64_t M, K, N, chunk;
  int32_t groups, mode;
  float eps;
  uint8_t* ws;
  HostWs wl;
  DeviceInfo dev;
  Planes wp{};

  int64_t rows_of(int64_t i) const { return (M - i * chunk) < chunk ? (M - i * chunk) : chunk; }

  bool setup() override { return start() && prepare_operand(W, N, K, mode, ws + wl.w_planes, dev, s, &wp) == GF_OK; }
  bool copy_in(int64_t i, int buf) override {
    return copy_in_bytes(buf, ws + wl.x[buf], x_host + size_t(i * chunk) * K, size_t(rows_of(i)) * K * 4);
  }
  bool compute(int64_t i, int buf) override {
    if (!compute_begin(buf)) return false;
    const int64_t rows = rows_of(i);
    const float* xd = reinterpret_cast<const float*>(ws + wl.x[buf]);
    float* od = reinterpret_cast<float*>(ws + wl.out[buf]);
    Planes xp{};
    const GNParams ep{b_lin, bias, gamma, beta, od, int(rows), int(N), eps, int(N / groups)};
    // (W's planes serve every chunk; a chunk's GEMM may compute x's lo plane
    // itself, lo_mask_at)
    return with_gn_epilogue(ep, s, [&](auto tag) {
             using E = typename decltype(tag)::type;
             const int lo = lo_mask_at<E>(mode, gemm_tile_width<E>(rows, N, mode, dev.sm_count));
             const gf_status st = prepare_operand(xd, rows, K, mode, ws + wl.xp[buf], dev, s, &xp, !(lo & 1));
             return st != GF_OK ? st : run_linear<E>(mode, dev, xp, wp, rows, kpad(K, mode), N, 0, ep, s);
           }) == GF_OK &&
           compute_end(buf);
  }
  bool copy_out(int64_t i, int buf) override {
    return copy_out_bytes(buf, out_host + size_t(i * chunk) * N, ws + wl.out[buf], size_t(rows_of(i)) * N * 4);
  }
};

// A stand-in for the CUDA side that records each step and fails at a chosen
// one (gf_testing_host_pipeline_trace).
struct TraceHostPipe final : HostPipeOps {
  int fail_at;  // index of the step that fails (-1: none)
  int step = 0;
  char* buf;
  size_t cap, len = 0;
  TraceHostPipe(int f, char* b, size_t c) : fail_at(f), buf(b), cap(c) {
    if (buf && cap) buf[0] = 0;
  }
  void put(const char* name, int64_t i) {
    char item[48];
    const int n = i < 0 ? std::snprintf(item, sizeof item, "%s%s", len ? " " : "", name)
                        : std::snprintf(item, sizeof item, "%s%s%lld", len ? " " : "", name, (long long)i);
    if (buf && n > 0 && len + size_t(n) < cap) {
      std::memcpy(buf + len, item, size_t(n) + 1);
      len += size_t(n);
    }
  }
  bool next(const char* name, int64_t i) {
    put(name, i);
    return step++ != fail_at;
  }
  bool setup() override { return next("setup", -1); }
  bool copy_in(int64_t i, int) override { return next("in", i); }
  bool compute(int64_t i, int) override { return next("compute", i); }
  bool copy_out(int64_t i, int) override { return next("out", i); }
  bool join() override { return next("join", -1); }
  void drain() override { put("drain", -1); }
};

}  // namespace

size_t gf_linear_swish_bias_groupnorm_host_workspace_size(int64_t M, int64_t K, int64_t N, int32_t groups,
                                                          int32_t mode, int64_t chunk_rows) {
  if (!mode_ok(mode) || check_linear_shape(M, K, N, mode) != GF_OK || !gn_groups_ok(N, groups) || chunk_rows < 0 ||
      M == 0)
    return 0;
  if (chunk_rows == 0) {
    DeviceInfo dev;
    if (current_device(&dev) != GF_OK) return 0;
    chunk_rows = host_chunk_rows(M, N, dev.sm_count);
  }
  return host_ws(chunk_rows < M ? chunk_rows : M, K, N, mode).total;
}

gf_status gf_linear_swish_bias_groupnorm_host(const float* x_host, const float* W, const float* b_lin,
                                              const float* bias, const float* gamma, const float* beta,
                                              float* out_host, int64_t M, int64_t K, int64_t N, int32_t groups,
                                              float eps, int32_t mode, int64_t chunk_rows, void* workspace,
                                              size_t workspace_bytes, void* stream) {
  if ((M && (!x_host || !out_host)) || !W || !bias || !gamma || !beta) return GF_ERR_NULL;
  if (!mode_ok(mode)) return GF_ERR_MODE;
  gf_status st = check_linear_shape(M, K, N, mode);
  if (st != GF_OK) return st;
  if (!gn_groups_ok(N, groups) || chunk_rows < 0) return GF_ERR_SHAPE;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return GF_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(bias) || !aligned16(gamma) || !aligned16(beta) ||
      (b_lin && !aligned16(b_lin)) || !aligned16(workspace))
    return GF_ERR_ALIGN;
  if (M == 0) return GF_OK;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != GF_OK) return st;
  const int64_t chunk = chunk_rows == 0 ? host_chunk_rows(M, N, dev.sm_count) : (chunk_rows < M ? chunk_rows : M);
  const HostWs wl = host_ws(chunk, K, N, mode);
  if (!workspace) return GF_ERR_NULL;
  if (workspace_bytes < wl.total) return GF_ERR_WORKSPACE;
  const Span ins[] = {{W, size_t(N) * K * 4}, {b_lin, size_t(N) * 4}, {bias, size_t(N) * 4},
                      {gamma, size_t(N) * 4}, {beta, size_t(N) * 4}};
  if ((st = check_no_alias(Span{workspace, wl.total}, ins, 5)) != GF_OK) return st;

  CudaHostPipe pipe;
  pipe.x_host = x_host;
  pipe.out_host = out_host;
  pipe.W = W;
  pipe.b_lin = b_lin;
  pipe.bias = bias;
  pipe.gamma = gamma;
  pipe.beta = beta;
  pipe.M = M;
  pipe.K = K;
  pipe.N = N;
  pipe.chunk = chunk;
  pipe.groups = groups;
  pipe.mode = mode;
  pipe.eps = eps;
  pipe.ws = static_cast<uint8_t*>(workspace);
  pipe.wl = wl;
  pipe.dev = dev;
  pipe.s = static_cast<cudaStream_t>(stream);
  if (!pipe.create()) return GF_ERR_CUDA;  // nothing enqueued yet
  return run_host_pipeline(pipe, (M + chunk - 1) / chunk);
}

gf_status gf_testing_host_pipeline_trace(int64_t nchunks, int32_t fail_at, char* trace, size_t trace_bytes) {
  if (nchunks < 0) return GF_ERR_SHAPE;
  TraceHostPipe pipe(fail_at, trace, trace_bytes);
  return run_host_pipeline(pipe, nchunks);
}

size_t gf_linear_workspace_size(int64_t M, int64_t K, int64_t N, int32_t mode) {
  if (!mode_ok(mode) || check_linear_shape(M, K, N, mode) != GF_OK || M == 0) return 0;
  return operand_ws_bytes(M, K, mode) + operand_ws_bytes(N, K, mode);
}

gf_status gf_linear(const float* x, const float* W, const float* b, float* out, int64_t M, int64_t K, int64_t N,
                    int32_t mode, void* workspace, size_t workspace_bytes, void* stream) {
  if ((M && (!x || !out)) || !W) return GF_ERR_NULL;
  if (!mode_ok(mode)) return GF_ERR_MODE;
  gf_status st = check_linear_shape(M, K, N, mode);
  if (st != GF_OK) return st;
  if (!aligned16(x) || !aligned16(W) || !aligned16(out) || (b && !aligned16(b)) || !aligned16(workspace))
    return GF_ERR_ALIGN;
  if (M == 0) return GF_OK;
  const size_t need = gf_linear_workspace_size(M, K, N, mode);
  if (!workspace) return GF_ERR_NULL;
  if (workspace_bytes < need) return GF_ERR_WORKSPACE;
  const Span ins[] = {{x, size_t(M) * K * 4}, {W, size_t(N) * K * 4}, {b, size_t(N) * 4}, {workspace, need}};
  st = check_no_alias(Span{out, size_t(M) * N * 4}, ins, 4);
  if (st != GF_OK) return st;
  EpiStore::Params ep{b, out, int(M), int(N)};
  return split_and_run<EpiStore>(mode, x, W, M, K, N, workspace, /*m_fastest=*/0, ep,
                                 static_cast<cudaStream_t>(stream));
}

size_t gf_linear_lse_act_workspace_size(int64_t M, int64_t K, int64_t N, int32_t mode) {
  if (!mode_ok(mode) || check_linear_shape(M, K, N, mode) != GF_OK || M == 0) return 0;
  // one (max, sum) partial per row and epilogue column half of each n-block,
  // sized for the narrowest tile width
  const int64_t nb = lse_parts(N, kLseWidths[0]);
  return operand_ws_bytes(M, K, mode) + operand_ws_bytes(N, K, mode) +
         align_up(size_t(M) * nb * sizeof(float2), 256);
}

gf_status gf_linear_lse_act(const float* x, const float* W, const float* b, float* out, int64_t M, int64_t K,
                            int64_t N, float negative_slope, int32_t mode, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if ((M && (!x || !out)) || !W) return GF_ERR_NULL;
  if (!mode_ok(mode)) return GF_ERR_MODE;
  gf_status st = check_linear_shape(M, K, N, mode);
  if (st != GF_OK) return st;
  if (!std::isfinite(negative_slope)) return GF_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(W) || !aligned16(out) || (b && !aligned16(b)) || !aligned16(workspace))
    return GF_ERR_ALIGN;
  if (M == 0) return GF_OK;
  const size_t need = gf_linear_lse_act_workspace_size(M, K, N, mode);
  if (!workspace) return GF_ERR_NULL;
  if (workspace_bytes < need) return GF_ERR_WORKSPACE;
  const Span ins[] = {{x, size_t(M) * K * 4}, {W, size_t(N) * K * 4}, {b, size_t(N) * 4}, {workspace, need}};
  st = check_no_alias(Span{out, size_t(M) * 4}, ins, 4);
  if (st != GF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float2* part = reinterpret_cast<float2*>(ws + operand_ws_bytes(M, K, mode) + operand_ws_bytes(N, K, mode));
  DeviceInfo dev;
  if ((st = current_device(&dev)) != GF_OK) return st;
  const int nb = int(lse_parts(N, linear_tile_width(true, M, N, 0, mode, dev.sm_count)));
  EpiLSEPartial::Params ep{b, part, int(M), int(N), nb};
  // m-blocks fastest: the CTAs in flight share n-blocks, so each W tile is
  // fetched from HBM once and reused by every m-block from L2.
  if ((st = split_and_run<EpiLSEPartial>(mode, x, W, M, K, N, workspace, /*m_fastest=*/1, ep, s)) != GF_OK)
    return st;
  const int threads = 256;
  const int blocks = int((M * 32 + threads - 1) / threads);
  lse_merge_act_kernel<<<blocks, threads, 0, s>>>(part, out, int(M), nb, negative_slope);
  return cuda_status(cudaGetLastError());
}

}  // extern "C"
