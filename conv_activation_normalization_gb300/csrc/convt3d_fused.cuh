// ConvTranspose3d(k 3, stride 2, pad 1) -> Swish -> GroupNorm -> HardSwish in
// one persistent kernel, the contraction on tcgen05 with the tiles, producer
// warps and MMA issuer of convt3d_tc.cuh.
//
// GroupNorm needs the statistics of a whole sample before any of its outputs
// can be written.  The two-pass kernels therefore run the contraction twice.
// Here every CTA keeps the Swish values of its last tiles in tensor memory
// instead, and the CTAs (all resident: cooperative launch, one per SM)
// exchange the statistics through global memory:
//
//   round r      CTA b of G computes tile t = r*G + b: MMA into TMEM buffer
//                r % 4, Swish, s written back over the accumulator
//                (tcgen05.st); the tile's per-group (sum s, sum s^2) go to
//                the tile's own slot in global memory and the sample's
//                counter of finished tiles is incremented;
//   round r + 3  (first thing in the round) once all tiles of t's sample are
//                counted, the CTA sums their slots (in a fixed order,
//                double-float arithmetic), turns the totals into the
//                per-channel affine (A, B) and writes tile t,
//                HardSwish(A s + B), straight from TMEM; that frees buffer
//                r % 4 for the MMAs of tile r + 4.
//
// A sample's tiles are consecutive, so with at most G + 1 tiles per sample it
// is complete at most one round after any of its tiles.  Between a CTA's own
// statistics of round r + 1 and its output of tile r lie the output of tile
// r - 1 and the statistics work of round r + 2, which hide the wait for the
// other CTAs; four 128-column TMEM buffers (all 512 columns) hold tiles
// r + 1 .. r + 3 and the MMA's target r + 4.  The host uses the two-pass
// kernels when a sample has more tiles than that.
//
// The weights (and the conv bias) are scaled by log2 e when the B tile is
// built, so the accumulator holds u = y log2 e and the Swish needs no scaling
// multiply: s' = u / (1 + 2^-u) = s log2 e.  GroupNorm of s' with
// eps (log2 e)^2 is exactly GroupNorm of s with eps (a common scale of the
// values and of sqrt(eps) cancels).
//
// Roles (768 threads):
//   warps 0-3    producers (thread = cell: gathers, A rows, and the cell's
//                record: output offset and which of its phases exist), warp 4
//                TMEM owner and MMA issuer (as in the two-pass kernel, with 4
//                accumulator buffers);
//   warp 5       publisher: per round, sums the epilogue warps' partial sums
//                into the tile's slot and counts the tile for its sample;
//   warps 6-7    coefficients, alternate tiles: waits (bounded) until every
//                tile of the tile's sample is counted, reduces the sample's
//                slots and writes the tile's 16 (A, A, B, B) into a shared
//                slot (two warps, so that one's reduction latency does not
//                limit the round rate);
//   warps 8-15   output: warp (8 + e) owns TMEM lane quadrant (warp % 4) and
//                the 64 columns of chunks 2 (e / 4) and 2 (e / 4) + 1 (chunk
//                c: output phases pd = c / 2, ph = c % 2, 16 channels x both
//                pw); per round it writes the tile from three rounds earlier;
//   warps 16-23  statistics: the same lanes and columns of the new tile,
//                a chunk per TMEM load: Swish, written back over the
//                accumulator, and the per-group sums.
// The two groups wait on different things (the coefficients and the Swish
// values of an old tile; the accumulator and the records of the new one), so
// each group's waits overlap the other's column work; they poll (the
// fastest wake-up measured here).  The Swish values cross from one group to
// the other through TMEM: a statistics warp waits for its tcgen05.st to
// complete and arrives on the buffer's `sdone` barrier, which the output
// warps wait on before their tcgen05.ld.
#pragma once

#include "convt3d_tc.cuh"

namespace gf {

constexpr int kCfEpiWarps = 16;
// Two output and two statistics warps per TMEM lane quadrant, each taking two
// of the quadrant's four 32-column chunks (one output warp and three
// statistics warps per quadrant took 0.297 ms per call against 0.239).
constexpr int kCfOutWarps = 8;   // warps 8-15
constexpr int kCfStatWarps = 8;  // warps 16-23
constexpr int kCfPubWarp = 5;
constexpr int kCfCoefWarp0 = 6;   // and 7
constexpr int kCfCoefWarps = 2;
constexpr int kCfEpiWarp0 = 8;
constexpr int kCfThreads = (kCfEpiWarp0 + kCfEpiWarps) * 32;
constexpr int kCfBufs = 4;                          // TMEM tile buffers of 128 columns
constexpr int kCfLag = 3;                           // rounds between a tile's statistics and its output
constexpr int kCfCoefFloats = 16 * 4;               // per buffer: 16 channels x (A, A, B, B)
constexpr int kCfPartFloats = kCfStatWarps * 8;     // per round: 8 sums per statistics warp
constexpr float kLog2e = 1.4426950408889634f;
// The producers run at most kCtTcStages tiles ahead of the MMAs, which run at
// most kCfBufs tiles ahead of the output of a tile: the records of the last
// 8 tiles cover that.
static_assert(kCtRecSlots >= kCtTcStages + kCfBufs, "record ring too short");
constexpr int kCfRecBytes = kCtRecSlots * 128 * 8;
constexpr int kCfSmem = kCtTcStages * kCtTcStageBytes + kCtTcBBytes + kCfBufs * kCfCoefFloats * 4 +
                        2 * kCfPartFloats * 4 + kCfRecBytes + 1024 /*barriers*/ + 1024 /*alignment*/;
static_assert(kCfOutWarps + kCfStatWarps == kCfEpiWarps, "the epilogue warps split into two groups");

struct CfParams {
  const float* x;
  const float* w;
  const float* bias;  // may be null
  const float* gamma;
  const float* beta;
  float* out;
  float* part;        // [num_tiles][8]: per tile and group g, (sum s', sum s'^2) at 2g, 2g + 1
  uint32_t* done;     // [N]: tiles of the sample whose slot is written; zero at launch
  int N, D, H, W;
  int bpp;            // tiles per (n, qd) plane: ceil(H*W / 128)
  int num_tiles;      // N * D * bpp
  int rounds;         // ceil(num_tiles / gridDim.x)
  FastDiv div_dp, div_bpp, div_w;  // by D * bpp (tiles per sample), bpp and W
  double inv_count;   // 1 / elements per (sample, group)
  float eps;          // GroupNorm eps x (log2 e)^2 (the statistics are of s')
  uint32_t plane;     // output elements per (sample, channel); 16 * plane < 2^32
  int OHW, OW;
};

// Wait until *cnt reaches `need`; false after the time limit.  Every lane
// polls with acquire loads, so each lane's later reads see what was written
// before the flag was raised.
__device__ __forceinline__ bool cf_wait_count(const uint32_t* cnt, uint32_t need) {
  if (ld_acquire_gpu(cnt) >= need) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    __nanosleep(64);
    if (ld_acquire_gpu(cnt) >= need) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Double-float arithmetic for the GroupNorm totals (fp64 is slow on this
// part): a value is an unevaluated sum hi + lo of two floats.
// Knuth's TwoSum: a + b = s + e exactly (round to nearest, no reassociation).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
// (hi, lo) += v
__device__ __forceinline__ void df_add(float& hi, float& lo, float v) {
  float e;
  two_sum(hi, v, hi, e);
  lo = __fadd_rn(lo, e);
}
// (hi, lo) += (h2, l2)
__device__ __forceinline__ void df_add2(float& hi, float& lo, float h2, float l2) {
  float e;
  two_sum(hi, h2, hi, e);
  lo = __fadd_rn(lo, __fadd_rn(e, l2));
}
// (hi, lo) * f with the product's rounding error kept (an FMA gives it exactly)
__device__ __forceinline__ void df_mul(float hi, float lo, float f, float& ph, float& pl) {
  ph = __fmul_rn(hi, f);
  pl = __fadd_rn(__fmaf_rn(hi, f, -ph), __fmul_rn(lo, f));
}

// The whole warp: sum the P tile slots of sample n (8 floats each) in a fixed
// order in double-float arithmetic and write the sample's per-channel affine
// A = gamma rsqrt(var + eps), B = beta - mean A, as (A, A, B, B), to
// coef[lane] (lane c < 16: channel c, group c / 4).  gam, bet: this lane's
// channel's gamma, beta.
__device__ __forceinline__ void cf_sample_coefs(const CfParams& p, int n, int P, int lane, float gam, float bet,
                                                float4* coef) {
  constexpr uint32_t kFull = 0xffffffffu;
  // lane l sums the float4 halves (l & 1) of tiles l / 2, l / 2 + 16, ...
  // (loads of a batch in flight together), then lanes of equal parity combine
  const float4* sp = reinterpret_cast<const float4*>(p.part + size_t(n) * P * 8);
  float h[4] = {0.f, 0.f, 0.f, 0.f}, l[4] = {0.f, 0.f, 0.f, 0.f};
  for (int i0 = 0; i0 < 2 * P; i0 += 8 * 32) {
    float4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + lane + 32 * j;
      v[j] = i < 2 * P ? __ldcg(sp + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      df_add(h[0], l[0], v[j].x);
      df_add(h[1], l[1], v[j].y);
      df_add(h[2], l[2], v[j].z);
      df_add(h[3], l[3], v[j].w);
    }
  }
  // reduce-scatter over the 16 lanes of equal parity (one half each): the
  // four values (s, s^2 of the half's first group, s, s^2 of its second)
  // split by lane bits 4 and 3, then the one kept value summed over bits 2
  // and 1; afterwards lane l holds value 2 b4 + b3 of half (l & 1)
  const bool b4 = lane & 16, b3 = lane & 8;
  float H[2], L[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float sh = b4 ? h[i] : h[2 + i], sl = b4 ? l[i] : l[2 + i];
    H[i] = b4 ? h[2 + i] : h[i];
    L[i] = b4 ? l[2 + i] : l[i];
    df_add2(H[i], L[i], __shfl_xor_sync(kFull, sh, 16), __shfl_xor_sync(kFull, sl, 16));
  }
  float vh = b3 ? H[1] : H[0], vl = b3 ? L[1] : L[0];
  {
    const float sh = b3 ? H[0] : H[1], sl = b3 ? L[0] : L[1];
    df_add2(vh, vl, __shfl_xor_sync(kFull, sh, 8), __shfl_xor_sync(kFull, sl, 8));
  }
#pragma unroll
  for (int o = 4; o >= 2; o >>= 1) df_add2(vh, vl, __shfl_xor_sync(kFull, vh, o), __shfl_xor_sync(kFull, vl, o));
  // channel lane c < 16: group g = c / 4 lies in half g / 2; its sum of s is
  // value 2 (g & 1), its sum of s^2 value 2 (g & 1) + 1
  const int g = (lane >> 2) & 3, s_src = (g >> 1) | ((g & 1) << 4), q_src = s_src | 8;
  const float s_h = __shfl_sync(kFull, vh, s_src), s_l = __shfl_sync(kFull, vl, s_src);
  const float q_h = __shfl_sync(kFull, vh, q_src), q_l = __shfl_sync(kFull, vl, q_src);
  if (lane < 16) {
    const float inv = float(p.inv_count);
    float mh, ml, qh, ql, ph, pl, vh2, ve;
    df_mul(s_h, s_l, inv, mh, ml);  // mean
    df_mul(q_h, q_l, inv, qh, ql);  // E[s^2]
    // mean^2 = mh^2 + 2 mh ml (+ ml^2, below the precision kept)
    ph = __fmul_rn(mh, mh);
    pl = __fadd_rn(__fmaf_rn(mh, mh, -ph), __fmul_rn(2.f * mh, ml));
    two_sum(qh, -ph, vh2, ve);
    const float var = fmaxf(__fadd_rn(vh2, __fadd_rn(ve, __fsub_rn(ql, pl))), 0.f);
    const float A = gam * rsqrtf(var + p.eps);
    const float B = bet - __fadd_rn(mh, ml) * A;
    coef[lane] = make_float4(A, A, B, B);
  }
}

// Columns 2 co + pw of a 32-column chunk are channel co at width phase pw;
// a chunk is one (pd, ph) output phase of all 16 channels.

// One chunk of an output warp: where its Swish values are, where its outputs
// go, and which of them exist.
struct CfOutSide {
  uint32_t taddr;     // TMEM address of the chunk's 32 columns (Swish values)
  float* oc;          // output of channel 0, width phase 0
  const float* cf;    // (A, A, B, B) per channel
  bool pv0, pv1;      // the width-phase-0 / 1 outputs lie inside the volume
};

// A statistics warp's work on one chunk of the new tile at q_taddr, its 32
// columns in one TMEM load: Swish of the accumulator values (u = y log2 e) in
// place, s' = u / (1 + 2^-u), written back over them; gs / gq get, per group,
// the (pw 0, pw 1) sums of s' and s'^2 (the caller masks out the phases that
// do not exist).  (A whole chunk per wait: 0.2391 -> 0.2348 ms per call
// against 16 columns.)
template <int K>
__device__ __forceinline__ void cf_stat_chunk(uint32_t q_taddr, const float* bias, float2 (&gs)[4],
                                              float2 (&gq)[4]) {
  uint32_t ry[32];
  GF_TMEM_LD32(q_taddr, ry);
  GF_TMEM_WAIT32(ry);
#pragma unroll
  for (int co = 0; co < 16; ++co) {
    const int g = co >> 2;
    float2 u = make_float2(__uint_as_float(ry[2 * co]), __uint_as_float(ry[2 * co + 1]));
    if constexpr (K == 32) {  // no padding column: the (scaled) bias is added here
      if (bias) {
        const float b = __ldg(bias + co) * kLog2e;
        u = add2(u, make_float2(b, b));
      }
    }
    const float2 d = add2(make_float2(ex2_approx(-u.x), ex2_approx(-u.y)), make_float2(1.f, 1.f));
    const float2 sv = mul2(u, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
    if ((co & 3) == 0) {
      gs[g] = sv;
      gq[g] = mul2(sv, sv);
    } else {
      gs[g] = add2(gs[g], sv);
      gq[g] = fma2(sv, sv, gq[g]);
    }
    ry[2 * co] = __float_as_uint(sv.x);
    ry[2 * co + 1] = __float_as_uint(sv.y);
  }
  GF_TMEM_ST32(q_taddr, ry);
}

// An output warp's round over its two chunks o[0], o[1] (the same 16
// channels at two (pd, ph) phases): per half of the channels, both chunks'
// 16 columns are loaded before one wait, and each channel's coefficients are
// read once for both; `tempty` is arrived on once every column is read.
// (Per call 0.2638 -> 0.2425 ms against one chunk at a time; doing the same on
// the statistics side, with its write-back, made it 0.253.)
__device__ __forceinline__ void cf_out_round(const CfOutSide (&o)[2], uint32_t plane, int lane, uint64_t* tempty) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t ra[16], rb[16];
    GF_TMEM_LD16(o[0].taddr + uint32_t(16 * h), ra);
    GF_TMEM_LD16(o[1].taddr + uint32_t(16 * h), rb);
    GF_TMEM_WAIT16(ra);
    GF_TMEM_WAIT16(rb);
    if (h == 1) {  // all columns read: the MMAs may overwrite the buffer
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int co = 8 * h + j;
      const float4 ab = reinterpret_cast<const float4*>(o[0].cf)[co];  // a broadcast read
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint32_t* r = k ? rb : ra;
        // GroupNorm affine A s' + B, then HardSwish h sat(h / 6 + 1/2); the
        // pair's two outputs are adjacent in memory
        const float2 sv = make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
        const float2 hv = fma2(make_float2(ab.x, ab.y), sv, make_float2(ab.z, ab.w));
        // (f32x2 FMAs have no saturating form)
        const float2 v = mul2(hv, make_float2(__saturatef(fmaf(hv.x, 1.f / 6.f, 0.5f)),
                                              __saturatef(fmaf(hv.y, 1.f / 6.f, 0.5f))));
        float* oc = o[k].oc + co * plane;  // (16 * plane < 2^32)
        if (o[k].pv0) __stcs(oc, v.x);
        if (o[k].pv1) __stcs(oc + 1, v.y);
      }
    }
  }
}

template <int CIN>
__global__ void __launch_bounds__(kCfThreads, 1) convt3d_fused_kernel(const CfParams p, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a_ring = smem;                                          // [S][hi, lo]
  uint8_t* b_tile = smem + kCtTcStages * kCtTcStageBytes;          // [hi, lo]
  float* coef_s = reinterpret_cast<float*>(b_tile + kCtTcBBytes);  // [kCfBufs][16][4]
  float* part_s = coef_s + kCfBufs * kCfCoefFloats;                // [2][kCfEpiWarps][8]
  uint64_t* rec_s = reinterpret_cast<uint64_t*>(part_s + 2 * kCfPartFloats);  // [kCtRecSlots][128]
  uint64_t* full = rec_s + kCtRecSlots * 128;
  uint64_t* empty = full + kCtTcStages;
  uint64_t* tfull = empty + kCtTcStages;  // accumulator of buffer b written by the MMAs
  uint64_t* tempty = tfull + kCfBufs;     // buffer b written out, free for the MMAs
  uint64_t* cfull = tempty + kCfBufs;     // coefficients of buffer b's tile ready
  uint64_t* cempty = cfull + kCfBufs;     // coefficient slot b read
  uint64_t* pfull = cempty + kCfBufs;     // [2] partial sums of the round written
  uint64_t* pempty = pfull + 2;           // [2] partial sums consumed
  uint64_t* rfull = pempty + 2;           // [kCtRecSlots] the tile's cell records written
  uint64_t* sdone = rfull + kCtRecSlots;  // [kCfBufs] buffer b's Swish values written back
  uint64_t* drain = sdone + kCfBufs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  constexpr int K = 8 * CIN;
  constexpr uint32_t kFull = 0xffffffffu;
  const int G = int(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kCtTcStages; ++s) {
      mbar_init(&full[s], kCtTcProducerThreads / 32);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < kCfBufs; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kCfOutWarps);
      mbar_init(&cfull[b], 1);
      mbar_init(&cempty[b], kCfOutWarps);
      mbar_init(&sdone[b], kCfStatWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&pfull[i], kCfStatWarps);
      mbar_init(&pempty[i], 1);
    }
    for (int i = 0; i < kCtRecSlots; ++i) mbar_init(&rfull[i], kCtTcProducerThreads / 32);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  ct_fill_tiles<CIN>(p.w, p.bias, a_ring, b_tile, kLog2e);
  fence_proxy_async_smem();
  if (warp == kCtTcMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kCfBufs * 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto fail = [&]() {
    record_error(status, GF_DEV_WAIT_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp < 4) {
    // ------------------------------------------------------------ producers
    const CtRecords rec{rec_s, rfull, uint64_t(p.plane), p.OHW, p.OW};
    ct_produce<CIN, true>(p, a_ring, full, empty, abort_flag, status, rec);
  } else if (warp == kCtTcMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0)
      ct_mma<kCfBufs, CIN>(p, tmem_base, a_ring, b_tile, full, empty, tfull, tempty, drain, abort_flag, status);
    __syncwarp();
  } else if (warp == kCfPubWarp) {
    // ----------------------------------------------------------- publisher
    bool ok = true;
    for (int r = 0; r < p.rounds; ++r) {
      const int t = blockIdx.x + r * G;
      if (!(ok = __all_sync(kFull, mbar_wait<true>(&pfull[r & 1], (r >> 1) & 1)) &&
                 !__any_sync(kFull, *abort_flag)))
        break;
      float v = 0.f;
      if (t < p.num_tiles && lane < 8) {
        // value v = lane: sum s' (even) or sum s'^2 (odd) of group lane / 2
        const float* ps = part_s + (r & 1) * kCfPartFloats + lane;
#pragma unroll
        for (int e = 0; e < kCfStatWarps; ++e) v += ps[e * 8];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&pempty[r & 1]);
      if (t < p.num_tiles) {
        if (lane < 8) p.part[size_t(t) * 8 + lane] = v;
        // release: the slot reaches L2 before the count says so
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(p.done + fdiv(t, p.div_dp), 1u);
      }
    }
    if (!ok) {
      fail();
      // the other CTAs must not wait for this one's tiles
      if (lane == 0)
        for (int n = 0; n < p.N; ++n) atomicAdd(p.done + n, 1u << 20);
    }
  } else if (warp < kCfEpiWarp0) {
    // -------------------------------------------------------- coefficients
    // warp kCfCoefWarp0 + i takes the tiles of rounds i, i + 2, ...; lane
    // c < 16: channel c's GroupNorm affine
    const int ci = warp - kCfCoefWarp0;
    const float gam = lane < 16 ? __ldg(p.gamma + lane) : 0.f, bet = lane < 16 ? __ldg(p.beta + lane) : 0.f;
    const int P = int(p.div_dp.d);
    for (int rt = ci; rt < p.rounds; rt += kCfCoefWarps) {
      const int t = blockIdx.x + rt * G;
      if (t >= p.num_tiles) break;
      const int slot = rt % kCfBufs, n = fdiv(t, p.div_dp);
      if (!__all_sync(kFull, mbar_wait<true>(&cempty[slot], ((rt / kCfBufs) & 1) ^ 1)) ||
          __any_sync(kFull, *abort_flag) || !__all_sync(kFull, cf_wait_count(p.done + n, uint32_t(P)))) {
        fail();
        break;
      }
      cf_sample_coefs(p, n, P, lane, gam, bet, reinterpret_cast<float4*>(coef_s + slot * kCfCoefFloats));
      __syncwarp();
      if (lane == 0) mbar_arrive(&cfull[slot]);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const bool out_group = warp < kCfEpiWarp0 + kCfOutWarps;
    const int e = out_group ? warp - kCfEpiWarp0 : warp - kCfEpiWarp0 - kCfOutWarps;
    const int quad = warp & 3, c0 = 2 * (e >> 2);  // the warp's chunks: c0, c0 + 1
    const int row = quad * 32 + lane;
    constexpr uint64_t kOffMask = (uint64_t(1) << 56) - 1;
    // record flags that make a chunk's width-phase-0 / 1 outputs exist: the
    // cell (bit 0), depth phase pd (bit 1), height phase ph (bit 2), width
    // phase 1 (bit 3)
    auto m0_of = [](int c) { return 1u | (uint32_t(c >> 1) << 1) | (uint32_t(c & 1) << 2); };
    const uint32_t lane_base = tmem_base + (uint32_t(quad * 32) << 16);
    if (out_group) {
      // ------------------------------------------------ output of old tiles
      for (int r = kCfLag; r < p.rounds + kCfLag; ++r) {
        if (__any_sync(kFull, *abort_flag)) break;
        const int ro = r - kCfLag, to = blockIdx.x + ro * G;
        if (to >= p.num_tiles) break;
        const int ob = ro % kCfBufs;
        // the tile's coefficients, its Swish values, and its records (the
        // slot's phase of round ro: its next use waits for this buffer)
        if (!__all_sync(kFull, mbar_wait(&cfull[ob], (ro / kCfBufs) & 1)) ||
            !__all_sync(kFull, mbar_wait(&sdone[ob], (ro / kCfBufs) & 1)) ||
            !__all_sync(kFull, mbar_wait(&rfull[ro % kCtRecSlots], (ro / kCtRecSlots) & 1))) {
          fail();
          break;
        }
        tc_fence_after();
        const uint64_t rv = rec_s[(ro % kCtRecSlots) * 128 + row];
        const uint32_t fl = uint32_t(rv >> 56);
        CfOutSide o[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int c = c0 + k;
          const uint32_t m0 = m0_of(c), m1 = m0 | 8u;
          o[k].pv0 = (fl & m0) == m0;
          o[k].pv1 = (fl & m1) == m1;
          o[k].taddr = lane_base + uint32_t(c * 32 + ob * 128);
          o[k].oc = p.out + ((rv & kOffMask) + uint32_t(c >> 1) * uint32_t(p.OHW) + uint32_t(c & 1) * uint32_t(p.OW));
          o[k].cf = coef_s + ob * kCfCoefFloats;
        }
        cf_out_round(o, p.plane, lane, &tempty[ob]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&cempty[ob]);
      }
    } else {
      // -------------------------------------------- statistics of new tiles
      for (int r = 0; r < p.rounds; ++r) {
        if (__any_sync(kFull, *abort_flag)) break;
        const int tp = blockIdx.x + r * G;
        const bool has_p1 = tp < p.num_tiles;
        if (!__all_sync(kFull, mbar_wait(&pempty[r & 1], ((r >> 1) & 1) ^ 1))) {
          fail();
          break;
        }
        float rs[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rs[i] = 0.f;
        if (has_p1) {
          const int buf = r % kCfBufs;
          if (!__all_sync(kFull, mbar_wait(&rfull[r % kCtRecSlots], (r / kCtRecSlots) & 1)) ||
              !__all_sync(kFull, mbar_wait(&tfull[buf], (r / kCfBufs) & 1))) {
            fail();
            break;
          }
          tc_fence_after();
          const uint32_t fl = uint32_t(rec_s[(r % kCtRecSlots) * 128 + row] >> 56);
          // the warp's two chunks, one at a time (a rolled loop: 0.2427 ->
          // 0.2391 ms per call against the unrolled one)
#pragma unroll 1
          for (int c = c0; c < c0 + 2; ++c) {
            const uint32_t m0 = m0_of(c), m1 = m0 | 8u;
            // the cell's existing phases of this chunk only
            const float mx = (fl & m0) == m0 ? 1.f : 0.f, my = (fl & m1) == m1 ? 1.f : 0.f;
            float2 gs[4], gq[4];
            cf_stat_chunk<K>(lane_base + uint32_t(c * 32 + buf * 128), p.bias, gs, gq);
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              rs[2 * g] += fmaf(gs[g].y, my, gs[g].x * mx);
              rs[2 * g + 1] += fmaf(gq[g].y, my, gq[g].x * mx);
            }
          }
          // the Swish values are in TMEM before the output warps read them
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sdone[buf]);
          // reduce-scatter of the 8 sums over the warp's 32 lanes (9
          // shuffles): afterwards lane l holds the full sum of value
          // v = 4*b4 + 2*b3 + b2 (b_i = bit i of l), value v being the sum
          // s' (even v) or s'^2 (odd v) of group v / 2
          const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float send = b4 ? rs[i] : rs[4 + i];
            const float keep = b4 ? rs[4 + i] : rs[i];
            rs[i] = keep + __shfl_xor_sync(kFull, send, 16);
          }
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const float send = b3 ? rs[i] : rs[2 + i];
            const float keep = b3 ? rs[2 + i] : rs[i];
            rs[i] = keep + __shfl_xor_sync(kFull, send, 8);
          }
          {
            const float send = b2 ? rs[0] : rs[1];
            const float keep = b2 ? rs[1] : rs[0];
            rs[0] = keep + __shfl_xor_sync(kFull, send, 4);
          }
          rs[0] += __shfl_xor_sync(kFull, rs[0], 2);
          rs[0] += __shfl_xor_sync(kFull, rs[0], 1);
          if ((lane & 3) == 0) part_s[(r & 1) * kCfPartFloats + e * 8 + (lane >> 2)] = rs[0];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfull[r & 1]);
      }
    }
  }

  if (warp >= kCfEpiWarp0) tmem_wait_st();
  tc_fence_before();
  __syncthreads();
  if (warp == kCtTcMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kCfBufs * 128);
  }
}

}  // namespace gf
