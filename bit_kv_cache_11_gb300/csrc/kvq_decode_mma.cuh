// kvq_decode_mma.cuh — tensor-core decode attention for the pages' geometry:
// keys grouped per channel, values grouped per token, G = 32 (the
// configuration "Your KV cache doesn't have a bit problem, it has a geometry
// problem" recommends, section "What to Do with This").
//
// Work split, partials and merge follow decode_split_kernel (kvq_decode.cuh):
// every warp streams a contiguous range of units (an equal share of the cost,
// where each pair adds virtual units for the work of leaving it).  With
// G = 32 a sub-block is a whole block, so one bulk copy of block_bytes moves a
// unit into a stage; tail units stream their fp16 rows through the same
// stages (mma_tail_chunk tokens per unit).  The first unit a warp loads for a
// pair also brings that pair's fp16 queries into a per-stage slot, so a warp
// never waits on a global load when it enters a pair.
//
// Scores and value sums run on mma.sync m16n8k16 (fp16 inputs, fp32
// accumulation) with the packed codes themselves as the A operand:
//   scores  S[token][n] = sum_c A_K[token][c] * B_K[c][n]
//   values  O[c][n]     = sum_tok A_V[c][tok] * B_V[tok][n]
// columns n = 2*r + h: query head r of the GQA group, h = 0/1 the high/low
// fp16 halves of an fp32 operand (hi + lo keeps ~22 bits).
//
// A operand.  Codes are stored in fragment order (include/kvq.h); for 2 and 4 bits
// each lane's codes sit in its own words, placed so that an AND mask leaves
// two codes c at bits p and p + 16 of a register -- an fp16 subnormal pair of
// value c * 2^(p - 24), exact, with no constant to remove.  2-bit words give
// their eight registers from the word and the word shifted right by 8 (p = 0,
// 2, 4, 6 for the first row of a register pair, p + 2 for the row 8 below),
// 4-bit words their four (p = 0 and 4).  8-bit words hold two fp16-operand
// byte pairs each (rows g and g+8); integer codes become exact fp16 values
// through a byte permute (1024 + c) and one half2 subtraction of 1024, E4M3
// codes through the fp8-pair conversion.
// B operand.  The fp32 value (q_c * s_c for scores, p_j * s_j for values)
// times 2^(24 - p) for its k-slot (folded into the query once per pair, and
// into the probabilities as they are stored), times a power of two that keeps
// it inside fp16's range, split into hi + lo.  Rows 8 below (p + 2, or p + 4
// for 4-bit codes) come out 4x (16x) and are scaled back once.
//
// Online softmax.  Scores are in log2 units (the query carries scale * log2
// e).  The running maximum m is raised only when a block holds a score more
// than kLazyMax above it (and at a pair's first block); otherwise the block's
// weights exp2(s - m) are used as they are (at most 2^kLazyMax), which keeps
// the block maximum and its cross-lane reduction off the common path.  The
// merge weighs partials by their own m, so the result is the same softmax.
#pragma once

#include "kvq_decode.cuh"

namespace kvq {

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^e for e in [-126, 127] (exact).
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + e) << 23); }

// 2^x with the SFU (ex2.approx: relative error about 2^-22; 0 for -inf).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// floor(log2(x)) for a positive normal x; -127 for zero/subnormal.
__device__ __forceinline__ int ilog2f(float x) { return ((__float_as_int(x) >> 23) & 0xff) - 127; }

// Fragment-order words -> A registers of m16n8k16 (a0 = row g, k 2t..2t+1;
// a1 = row g+8, same k; a2 = row g, k 2t+8..2t+9; a3 = row g+8, same k).
// 2-bit word: k-step `half` (0 or 1) of the two k-steps it holds.
__device__ __forceinline__ void frag_a2(uint32_t w, int half, uint32_t& a0, uint32_t& a1,
                                        uint32_t& a2, uint32_t& a3) {
  const uint32_t y = w >> 8;
  if (half == 0) {
    a0 = w & 0x00030003u;  // p 0
    a1 = w & 0x000C000Cu;  // p 2
    a2 = y & 0x000C000Cu;  // p 2 (word bits 10-11)
    a3 = w & 0x00300030u;  // p 4
  } else {
    a0 = y & 0x00300030u;  // p 4 (word bits 12-13)
    a1 = w & 0x00C000C0u;  // p 6
    a2 = y & 0x00C000C0u;  // p 6 (word bits 14-15)
    a3 = w & 0x03000300u;  // p 8
  }
}
// 4-bit word: one k-step.
__device__ __forceinline__ void frag_a4(uint32_t w, uint32_t& a0, uint32_t& a1, uint32_t& a2,
                                        uint32_t& a3) {
  const uint32_t y = w >> 8;
  a0 = w & 0x000F000Fu;  // p 0
  a1 = w & 0x00F000F0u;  // p 4
  a2 = y & 0x000F000Fu;  // p 0 (word bits 8-11)
  a3 = y & 0x00F000F0u;  // p 4 (word bits 12-15)
}

// 8-bit fragment-order words -> A registers of one k-step: word x.x holds
// row g (bytes 0-1) and row g+8 (bytes 2-3) at columns 2t, 2t+1; word x.y the
// same at columns 2t+8, 2t+9.  Integer codes become exact fp16 values through
// 1024 + c; E4M3 codes (F8) through the fp8-pair conversion, also exact.
template <bool F8>
__device__ __forceinline__ void frag_a8(uint2 x, uint32_t& a0, uint32_t& a1, uint32_t& a2,
                                        uint32_t& a3) {
  if constexpr (F8) {
    a0 = e4m3x2_to_half2(x.x);
    a1 = e4m3x2_to_half2(x.x >> 16);
    a2 = e4m3x2_to_half2(x.y);
    a3 = e4m3x2_to_half2(x.y >> 16);
  } else {
    const __half2 k1024 = __float2half2_rn(1024.0f);
    auto pair = [&](uint32_t v, uint32_t sel) -> uint32_t {
      uint32_t b = __byte_perm(v, 0x64646464u, sel);  // 1024 + byte, 1024 + byte
      __half2 h = __hsub2(*reinterpret_cast<__half2*>(&b), k1024);
      return *reinterpret_cast<uint32_t*>(&h);
    };
    a0 = pair(x.x, 0x4140u);
    a1 = pair(x.x, 0x4342u);
    a2 = pair(x.y, 0x4140u);
    a3 = pair(x.y, 0x4342u);
  }
}

// The two 8-bit words of (m-tile mt, k-step ks) of lane `lane` in a region of
// KSN k-steps per m-tile: words 2*(mt*KSN + ks) and the next, adjacent.
template <int KSN>
__device__ __forceinline__ uint2 words8(const uint32_t* region, int mt, int ks, int lane) {
  const int w = 2 * (mt * KSN + ks);
  return *reinterpret_cast<const uint2*>(region + ((w >> 2) * 32 + lane) * 4 + (w & 3));
}

// Largest value of the warp for non-negative finite x: the bit patterns of
// such floats order as unsigned integers, so one redux.sync finds it.
__device__ __forceinline__ float warp_max_nonneg(float x) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(x)));
}

// Weights exp2(s - m) of a block may reach 2^kLazyMax before m is raised.
constexpr float kLazyMax = 8.0f;

// log2 of the factor 2^(24 - p) of a value code at token tau (B_V operand):
// 2-bit codes sit at p = 2 (2 ((tau >> 4) & 1) + ((tau >> 3) & 1)), 4-bit codes
// at p = 0, 8-bit codes are exact fp16 values (factor 1).
template <int BV>
__host__ __device__ constexpr int vcode_log2(int tau) {
  return BV == 2 ? 24 - 2 * (2 * ((tau >> 4) & 1) + ((tau >> 3) & 1)) : (BV == 4 ? 24 : 0);
}

template <int D, int BK, int BV, int R, bool ROPE, bool OUT = false>
struct MmaCfg {
  static constexpr int G = 32;
  static constexpr int NG = D / 32;               // value channel groups
  static constexpr int MTV = D / 16;              // value m-tiles
  static constexpr int CPL = D / 32;              // output channels per lane
  static constexpr int NT = (2 * R + 7) / 8;      // n-tiles = query groups of 4
  static constexpr int KS = D / 16;               // key k-steps
  static constexpr int KP = D / 64;               // key channel pairs per lane
  static constexpr int VJ = NG / 2;               // value items per lane
  static constexpr int KWL = D * BK / 32;         // key words per lane / per row
  static constexpr int VWL = D * BV / 32;         // value words per lane (fragment)
  // rows 8 below come out this many times too large (fragment order)
  static constexpr float RK = BK == 2 ? 0.25f : (BK == 4 ? 0.0625f : 1.f);
  static constexpr float RV = BV == 2 ? 0.25f : (BV == 4 ? 0.0625f : 1.f);
  static constexpr int KC_S = 4 * D * BK;
  static constexpr int KM_S = 4 * D;
  static constexpr int VC_S = 4 * D * BV;
  static constexpr int VM_S = 4 * D;
  // Dense-and-sparse blocks (OUT) carry up to kMaxOut outlier entries per
  // side after each side's metadata: the stage holds the largest block and
  // the value sections sit 4 * nout bytes further (a runtime offset).
  static constexpr int kMaxOut = 64;
  static constexpr int BLK = KC_S + KM_S + VC_S + VM_S;    // a block without outliers
  // RoPE stages also carry the cos/sin row (D/2 float2) of the block's first
  // position, copied with the block.
  static constexpr int STAGE = BLK + (OUT ? 8 * kMaxOut : 0) + (ROPE ? 4 * D : 0);
  // Two stages where shared memory would otherwise limit the CTAs per SM
  // (RoPE tables, four or more query heads): more resident warps instead.
  static constexpr int NS = (ROPE || R >= 4) ? 2 : (STAGE <= 4096 ? 3 : 2);
  static constexpr int TCH = mma_tail_chunk(BK, BV);
  static constexpr int QB = R * D * 2;            // one pair's fp16 queries
  // B-operand blocks hold only the lanes whose columns exist: BL lanes
  // (columns < 2R of a single n-tile live in lanes < 8R), padded to BSTR
  // uint2 so that the lanes filling one column of several blocks at once hit
  // distinct banks (the block stride in words is an odd multiple of 8 banks
  // apart for the four blocks a store instruction touches).
  static constexpr int BL = NT == 1 ? (8 * R < 32 ? 8 * R : 32) : 32;
  static constexpr int BSTR = NT == 1 ? BL + 4 : BL + 2;
  static constexpr int OFF_BAR = NS * STAGE;
  static constexpr int OFF_QS = OFF_BAR + 64;                       // [NS][QB] query slots
  static constexpr int OFF_KB = OFF_QS + NS * QB;                   // [KS*NT][BSTR] uint2
  static constexpr int KB_BYTES = ROPE ? 0 : KS * NT * BSTR * 8;
  static constexpr int OFF_VB = OFF_KB + KB_BYTES;                  // [NG*2*NT][BSTR] uint2
  static constexpr int VB_BYTES = NG * 2 * NT * BSTR * 8;
  static constexpr int OFF_PB = OFF_VB + VB_BYTES;                  // [R][32] float
  static constexpr int OFF_OS = OFF_PB + R * 32 * 4;                // [R][D] float
  // RoPE: per-warp key coefficients, six per frequency pair, stored for
  // pairs (2f, 2f + 1) as three float4 [R][D/4][3]; per-CTA table of
  // cos/sin(j * theta_i), j < 32, stored [D/4][32] float4 {cos_2f, cos_2f+1,
  // sin_2f, sin_2f+1} so that lane j reads its own row conflict-free.
  static constexpr int OFF_CF = OFF_OS + R * D * 4;
  // OUT: score corrections [R][32] and value corrections [R][D] (floats)
  static constexpr int OFF_KX = OFF_CF + (ROPE ? R * (D / 4) * 48 : 0);
  static constexpr int OFF_VX = OFF_KX + (OUT ? R * 32 * 4 : 0);
  static constexpr int WARP_BYTES = round_up(OFF_VX + (OUT ? R * D * 4 : 0), 128);
  static constexpr int CS_BYTES = ROPE ? (D / 4) * 32 * 16 : 0;
  // Warps per CTA, and CTAs per SM the registers allow (the register budget
  // per thread is 65536 / (32 NW MINB)).
  // 8-bit sides on both halves (two 9 KB stages per warp): 5 warps in each of
  // two CTAs fill the shared memory (10 warps per SM instead of 8).
  static constexpr int NW = (BK == 8 && BV == 8 && R == 1 && !ROPE) ? 5 : 4;
  static constexpr int MINB = (BK == 8 && BV == 8 && R == 1 && !ROPE) ? 2 : (R <= 4 ? 3 : 1);
  static constexpr int SMEM = NW * WARP_BYTES + CS_BYTES;
  static_assert(2 * TCH * D * 2 == BLK, "a tail chunk fills a block's stage");
  static_assert(!(OUT && ROPE), "outlier corrections are applied to post-RoPE keys");
  static_assert(KWL % 4 == 0, "lane words are read as 16-byte vectors");
  static_assert(VWL % 4 == 0, "lane words are read as 16-byte vectors");
  static_assert(QB % 16 == 0 && OFF_QS % 16 == 0, "query slots are bulk-copy targets");
};

// Word offset, inside a B-operand region, of column n relative to column 0
// of the same lane slot (the slot's base holds its block, lane and register).
template <int BSTR>
__host__ __device__ constexpr int bcol(int n) {
  return (n >> 3) * BSTR * 2 + (n & 7) * 8;
}

template <int D, int BK, int BV, int R, bool ROPE, bool F8 = false, bool OUT = false>
__global__ void __launch_bounds__(MmaCfg<D, BK, BV, R, ROPE, OUT>::NW * 32,
                                  MmaCfg<D, BK, BV, R, ROPE, OUT>::MINB)
    decode_mma_kernel(const __grid_constant__ DecodeParams p) {
  using C = MmaCfg<D, BK, BV, R, ROPE, OUT>;
  constexpr int NS = C::NS, NT = C::NT, NG = C::NG, MTV = C::MTV, CPL = C::CPL, TCH = C::TCH,
                STAGE = C::STAGE, KS = C::KS, BL = C::BL, BSTR = C::BSTR, KP = C::KP,
                VJ = C::VJ, QB = C::QB;

  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int gw = blockIdx.x * C::NW + warp;
  // Up to griddepcontrol.wait below nothing reads or writes what the
  // preceding grid in the stream may still touch, so this runs while it
  // finishes: this warp's units [ua, ub), its barriers, load cursor and
  // per-lane constants.
  int ua = 0, ub = 0;
  if (gw < p.n_warps) warp_units(p.map, gw, &ua, &ub);
  const bool active = ua < ub;
  if (!active) ua = ub = 0;

  uint8_t* ws = smem + warp * C::WARP_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ws + C::OFF_BAR);
  uint32_t* kb32 = reinterpret_cast<uint32_t*>(ws + C::OFF_KB);
  uint32_t* vb32 = reinterpret_cast<uint32_t*>(ws + C::OFF_VB);
  const uint2* kbv = reinterpret_cast<const uint2*>(ws + C::OFF_KB);
  const uint2* vbv = reinterpret_cast<const uint2*>(ws + C::OFF_VB);
  float* pb = reinterpret_cast<float*>(ws + C::OFF_PB);
  float* os = reinterpret_cast<float*>(ws + C::OFF_OS);
  float* kx = reinterpret_cast<float*>(ws + C::OFF_KX);  // OUT: score corrections [R][32]
  float* vx = reinterpret_cast<float*>(ws + C::OFF_VX);  // OUT: value corrections [R][D]
  // a block's bytes, and where its value sections start in a stage
  const int nout = OUT ? p.g.nout : 0;
  const uint32_t blk_bytes = OUT ? static_cast<uint32_t>(p.g.block_bytes) : static_cast<uint32_t>(C::BLK);
  const int voff = C::KC_S + C::KM_S + 4 * nout;
  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  // ---- the load cursor (unit lj of pair lpr), NS units ahead of compute
  int lu = ua;
  int lpr = static_cast<int>(pair_of_unit(p.map, ua));
  int lj = ua - static_cast<int>(first_unit(p.map, lpr));
  int lnsub = pair_nsub(p, lpr), lupp = pair_upp(p, lpr);
  bool lfirst = true;  // the next load is this warp's first unit of its pair
  const uint8_t* lbase = p.g.blocks + static_cast<size_t>(lpr) * p.g.NB * blk_bytes;
  // Lane 0: unit (lpr, lj) -> stage s, plus the pair's queries into the
  // stage's query slot when it is the warp's first unit of the pair.
  auto issue = [&](int s) {
    uint8_t* st = ws + s * STAGE;
    const uint32_t qb = lfirst ? static_cast<uint32_t>(QB) : 0u;
    if (lj < lnsub) {
      mbar_arrive_expect_tx(&bars[s], blk_bytes + qb + (ROPE ? 4 * D : 0));
      bulk_g2s(st, lbase + static_cast<size_t>(lj) * blk_bytes, blk_bytes, &bars[s]);
      if constexpr (ROPE) {
        const int p0 = p.map.Ts[row_of(p.map, lpr)] + 32 * lj;
        bulk_g2s(st + C::BLK, p.rope_tab + static_cast<size_t>(p0) * (D / 2), 4 * D, &bars[s]);
      }
    } else {
      const PairLens ll = pair_lens(p, lpr);
      if (lj >= ll.nsub + ll.ntu) {
        // sink rows [t0, t1): K rows, then V rows, one copy each
        const int t0 = (lj - ll.nsub - ll.ntu) * TCH;
        const int t1 = min(t0 + TCH, ll.Ts);
        const uint32_t bytes = static_cast<uint32_t>(t1 - t0) * D * 2;
        const size_t row = static_cast<size_t>(lpr) * p.g.NSK + t0;
        mbar_arrive_expect_tx(&bars[s], 2 * bytes + qb);
        bulk_g2s(st, p.ksink + row * D, bytes, &bars[s]);
        bulk_g2s(st + TCH * D * 2, p.vsink + row * D, bytes, &bars[s]);
      } else {
        // tail rows [t0, t1): those below t_old from the tail buffer, the rest
        // (tokens appended by this call) from knew / vnew
        const int t0 = (lj - ll.nsub) * TCH;
        const int t1 = min(t0 + TCH, ll.Tt);
        const int tm = max(t0, min(t1, ll.t_old));
        mbar_arrive_expect_tx(&bars[s], static_cast<uint32_t>(t1 - t0) * D * 4 + qb);
        if (tm > t0) {
          const uint32_t bytes = static_cast<uint32_t>(tm - t0) * D * 2;
          const size_t row = static_cast<size_t>(lpr) * p.g.TC + t0;
          bulk_g2s(st, p.ktail[ll.buf] + row * D, bytes, &bars[s]);
          bulk_g2s(st + TCH * D * 2, p.vtail[ll.buf] + row * D, bytes, &bars[s]);
        }
        if (t1 > tm) {
          const int n_new = p.n_new;
          const uint32_t bytes = static_cast<uint32_t>(t1 - tm) * D * 2;
          const size_t row = static_cast<size_t>(lpr) * n_new + (tm - ll.t_old);
          bulk_g2s(st + (tm - t0) * D * 2, p.knew + row * D, bytes, &bars[s]);
          bulk_g2s(st + (TCH + tm - t0) * D * 2, p.vnew + row * D, bytes, &bars[s]);
        }
      }
    }
    if (qb) bulk_g2s(ws + C::OFF_QS + s * QB, p.q + static_cast<size_t>(lpr) * R * D, QB, &bars[s]);
  };
  auto advance_load = [&]() {
    ++lu;
    lfirst = false;
    if (++lj == lupp) {
      lj = 0;
      ++lpr;
      lfirst = true;
      lbase += static_cast<size_t>(p.g.NB) * blk_bytes;
      if (lu < ub) {
        lnsub = pair_nsub(p, lpr);
        lupp = pair_upp(p, lpr);
      }
    }
  };
  // ---- per-lane constants of the B operands
  // Keys: channel pairs P = lane + 32 i (k-step ks = P >> 3, register
  // rg = (P >> 2) & 1, lane slot t); channels kch[i], kch[i] + 1.
  const int rg = (lane >> 2) & 1;
  int kch[KP], kbo[KP];
#pragma unroll
  for (int i = 0; i < KP; ++i) {
    const int ks = (lane >> 3) + 4 * i;
    kch[i] = 16 * ks + 8 * rg + 2 * t;
    kbo[i] = ks * NT * BSTR * 2 + 2 * t + rg;
  }
  // code factor 2^(24 - p) of the lane's key slots (the same for every i)
  const int klog = BK == 2 ? 24 - 2 * (2 * ((lane >> 3) & 1) + rg) : (BK == 4 ? 24 : 0);
  const float kf = pow2i(klog), kfinv = pow2i(-klog);
  // Values: items J = lane + 32 i: token pair J & 15 (tokens tau0, tau0 + 1),
  // channel group (lane >> 4) + 2 i.
  const int ksv = (lane >> 3) & 1;
  const int tau0 = 16 * ksv + 8 * rg + 2 * t;
  int vbo[VJ];
#pragma unroll
  for (int i = 0; i < VJ; ++i) vbo[i] = (((lane >> 4) + 2 * i) * 2 + ksv) * NT * BSTR * 2 + 2 * t + rg;
  const float vfinv = pow2i(-vcode_log2<BV>(tau0));  // the lane's items' code factor, inverted
  const float vfl = pow2i(vcode_log2<BV>(lane));      // code factor of token `lane`

  // Operand buffers: columns that no query fills stay zero; lanes >= BL
  // (no column of theirs exists) read the zeroed padding slots of a block.
  for (int i = lane; i < (C::OFF_PB - C::OFF_KB) / 4; i += 32) kb32[i] = 0u;
  static_assert(BL == 32 || BSTR >= BL + 4, "padding slots for the lanes beyond BL");
  const int blane = lane < BL ? lane : BL + (lane & 3);
  __syncwarp();

  // Launched as a programmatic dependent: wait until the preceding grid in
  // the stream has completed (and its writes are visible) before touching
  // global memory, and let the next grid launch while this one runs.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // RoPE: cos/sin(j * theta_i) for the 32 token offsets of a sub-block (table
  // rows 0..31), transposed so lane j reads its own column conflict-free, two
  // frequency pairs per entry.  Loaded before any warp of the CTA can leave.
  float4* cs_tab = reinterpret_cast<float4*>(smem + C::NW * C::WARP_BYTES);
  if constexpr (ROPE) {
    for (int idx = threadIdx.x; idx < (D / 4) * 32; idx += blockDim.x) {
      const int f = idx >> 5, j = idx & 31;
      const bool in = j < p.rope_rows;
      const float2 a = in ? p.rope_tab[static_cast<size_t>(j) * (D / 2) + 2 * f] : make_float2(1.f, 0.f);
      const float2 b = in ? p.rope_tab[static_cast<size_t>(j) * (D / 2) + 2 * f + 1] : make_float2(1.f, 0.f);
      cs_tab[idx] = make_float4(a.x, b.x, a.y, b.y);
    }
    __syncthreads();
  }
  // Fused append: store the new tokens into the tail for later calls (no
  // access of this launch reads those tail rows).
  if (p.n_new > 0) {
    const int n_new = p.n_new;
    const long long chunks = static_cast<long long>(p.g.P) * n_new * (D / 8);
    for (long long c = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; c < chunks;
         c += static_cast<long long>(gridDim.x) * blockDim.x) {
      const long long rowi = c / (D / 8);
      const int col = static_cast<int>(c - rowi * (D / 8)) * 8;
      const long long pr = rowi / n_new;
      const int r = static_cast<int>(rowi - pr * n_new);
      const int b = row_of(p.map, pr);
      const int buf = static_cast<int>((p.act >> b) & 1ull);
      const size_t dst = (static_cast<size_t>(pr) * p.g.TC + (p.map.Tt[b] - n_new) + r) * D + col;
      *reinterpret_cast<uint4*>(p.ktail[buf] + dst) =
          *reinterpret_cast<const uint4*>(p.knew + rowi * D + col);
      *reinterpret_cast<uint4*>(p.vtail[buf] + dst) =
          *reinterpret_cast<const uint4*>(p.vnew + rowi * D + col);
    }
  }
  if (!active) return;
  for (int s = 0; s < NS && lu < ub; ++s) {
    if (lane == 0) issue(s);
    advance_load();
  }

  // ---- state of the current pair
  float qf[R][KP][2];    // q * scale * log2(e) * 2^klog of this lane's key channels
  float m[R];            // running maximum (log2 units), identical in all lanes
  float mlk[NT][4];      // m of the lane's query minus log2 f of its four score tokens
  float lq[R];           // this lane's share of the softmax denominators
  float acc[MTV][NT][4];
  float corr[R][VJ];     // value zero-point sums of this lane's items (in units of the code factor)
  float acct[R][CPL];    // fp16-tail contributions, channels lane*CPL + c
  int ev = -126;         // value operand exponent: B_V = p * s * f * 2^-ev
  int cur = -1;

  // value of f for this lane's query column (query 4*nt + t), 1 if none
  auto lane_factor = [&](const float (&f)[R], int nt) -> float {
    float v = 1.f;
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (r == 4 * nt + t) v = f[r];
    return v;
  };

  auto set_mlk = [&]() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float mq = lane_factor(m, nt);
#pragma unroll
      for (int k = 0; k < 4; ++k) mlk[nt][k] = mq - static_cast<float>(vcode_log2<BV>(8 * k));
    }
  };

  // New pair: its queries from the query slot of stage s.
  auto enter_pair = [&](int s) {
    const __half* qp = reinterpret_cast<const __half*>(ws + C::OFF_QS + s * QB);
    if constexpr (!ROPE) {
#pragma unroll
      for (int i = 0; i < KP; ++i)
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float2 q2 = __half22float2(*reinterpret_cast<const __half2*>(qp + r * D + kch[i]));
          const float sc = p.qscale * kf;
          qf[r][i][0] = q2.x * sc;
          qf[r][i][1] = q2.y * sc;
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      m[r] = -INFINITY;
      lq[r] = 0.f;
#pragma unroll
      for (int k = 0; k < VJ; ++k) corr[r][k] = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) acct[r][c] = 0.f;
    }
    set_mlk();
#pragma unroll
    for (int a = 0; a < MTV; ++a)
#pragma unroll
      for (int b = 0; b < NT; ++b)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[a][b][k] = 0.f;
    ev = -126;
    // the scaled query, all channels (rotated-key sub-blocks and the tail)
    for (int i = lane; i < R * D; i += 32) os[i] = __half2float(qp[i]) * p.qscale;
    if constexpr (OUT)
      for (int i = lane; i < R * D; i += 32) vx[i] = 0.f;
    __syncwarp();
  };

  // The running maximum rose: multiply everything accumulated by alpha.
  auto rescale_all = [&](const float (&alpha)[R]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float lf = lane_factor(alpha, nt);
#pragma unroll
      for (int a = 0; a < MTV; ++a)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[a][nt][k] *= lf;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      lq[r] *= alpha[r];
#pragma unroll
      for (int k = 0; k < VJ; ++k) corr[r][k] *= alpha[r];
#pragma unroll
      for (int c = 0; c < CPL; ++c) acct[r][c] *= alpha[r];
      if constexpr (OUT) {
        __syncwarp();
        for (int i = lane; i < D; i += 32) vx[r * D + i] *= alpha[r];
        __syncwarp();
      }
    }
  };

  // Eager update of the running maximum to the block maxima mx; rescales
  // when it rises.
  auto raise_max = [&](const float (&mx)[R]) {
    float alpha[R];
    bool any = false;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float mn = fmaxf(m[r], mx[r]);
      any |= mn != m[r];
      alpha[r] = fast_exp2(m[r] - mn);
      m[r] = mn;
    }
    if (any) {  // warp-uniform
      rescale_all(alpha);
      set_mlk();
    }
  };

  // ---- pieces of a sub-block (keys stored after RoPE), so that the main
  // loop can put the key mma of one block and the value mma of the previous
  // block in one basic block (two independent instruction streams).
  auto k_prep = [&](const uint8_t* st, float (&kz)[R], float& ek2) {
    // ---- key operand: B_K[c][2r+h] = hi/lo of q_r[c] s_c f_c 2^-ek
    float qh[R][KP][2];
    float kzl[R];
    float amax = 0.f;
#pragma unroll
    for (int r = 0; r < R; ++r) kzl[r] = 0.f;
#pragma unroll
    for (int i = 0; i < KP; ++i) {
      // {scale, zero} of channels kch[i] and kch[i] + 1
      const uint2 mm = *reinterpret_cast<const uint2*>(st + C::KC_S + 4 * kch[i]);
      const float2 s0 = __half22float2(*reinterpret_cast<const __half2*>(&mm.x));
      const float2 s1 = __half22float2(*reinterpret_cast<const __half2*>(&mm.y));
#pragma unroll
      for (int r = 0; r < R; ++r) {
        qh[r][i][0] = qf[r][i][0] * s0.x;
        qh[r][i][1] = qf[r][i][1] * s1.x;
        kzl[r] = fmaf(qf[r][i][0], s0.y, fmaf(qf[r][i][1], s1.y, kzl[r]));
        amax = fmaxf(amax, fmaxf(fabsf(qh[r][i][0]), fabsf(qh[r][i][1])));
      }
    }
    amax = warp_max_nonneg(amax);
    // |B| < 2^14: one exponent for the sub-block
    const int ek = min(max(ilog2f(amax) - 13, -120), 120);
    const float sk = pow2i(-ek);
    ek2 = pow2i(ek);
#pragma unroll
    for (int i = 0; i < KP; ++i) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float v0 = qh[r][i][0] * sk, v1 = qh[r][i][1] * sk;
        const __half2 hi = __floats2half2_rn(v0, v1);
        const float2 hf = __half22float2(hi);
        const __half2 lo = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
        kb32[kbo[i] + bcol<BSTR>(2 * r)] = *reinterpret_cast<const uint32_t*>(&hi);
        kb32[kbo[i] + bcol<BSTR>(2 * r + 1)] = *reinterpret_cast<const uint32_t*>(&lo);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) kz[r] = warp_sum(kzl[r] * kfinv);
    __syncwarp();
  };

  auto k_mma = [&](const uint8_t* st, float (&sc)[2][NT][4]) {
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(st);
    // ---- scores: tokens 16*mt + g (c0,c1) and 16*mt + g + 8 (c2,c3); even
    // and odd k-steps accumulate apart (four independent mma chains), then add
    float sa[2][2][NT][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int b = 0; b < NT; ++b)
#pragma unroll
          for (int k = 0; k < 4; ++k) sa[a][h][b][k] = 0.f;
    if constexpr (BK == 8) {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          uint32_t a0, a1, a2, a3;
          frag_a8<F8>(words8<KS>(kc, mt, ks, lane), a0, a1, a2, a3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint2 b = kbv[(ks * NT + nt) * BSTR + blane];
            mma_16816(sa[mt][ks & 1][nt], a0, a1, a2, a3, b.x, b.y);
          }
        }
    } else {
      uint32_t kw[C::KWL];
#pragma unroll
      for (int q = 0; q < C::KWL / 4; ++q) {
        const uint4 x = reinterpret_cast<const uint4*>(kc)[q * 32 + lane];
        kw[4 * q] = x.x; kw[4 * q + 1] = x.y; kw[4 * q + 2] = x.z; kw[4 * q + 3] = x.w;
      }
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          uint32_t a0, a1, a2, a3;
          if constexpr (BK == 2) frag_a2(kw[mt * (KS / 2) + (ks >> 1)], ks & 1, a0, a1, a2, a3);
          else frag_a4(kw[mt * KS + ks], a0, a1, a2, a3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint2 b = kbv[(ks * NT + nt) * BSTR + blane];
            mma_16816(sa[mt][ks & 1][nt], a0, a1, a2, a3, b.x, b.y);
          }
        }
    }
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < NT; ++b)
#pragma unroll
        for (int k = 0; k < 4; ++k) sc[a][b][k] = sa[a][0][b][k] + sa[a][1][b][k];
  };

  // Scores -> weights of the block (lazy maximum), stored in pb with each
  // token's value code factor folded in; the lane's shares of l grow.
  auto softmax_scores = [&](const uint8_t* st, float (&sc)[2][NT][4], const float (&kz)[R],
                            float ek2) {
    // lane holds query 4*nt + t, tokens g, g + 8, g + 16, g + 24 (s4[nt][k])
    float s4[NT][4];
    float dmax = -INFINITY;
    if constexpr (OUT) {
      // kept key outliers: the dense path scored them as their group's zero
      // point; token j gains q_c (x - z_c) for each kept (j, c)
      const __half2* km = reinterpret_cast<const __half2*>(st + C::KC_S);
      const uint32_t* ko = reinterpret_cast<const uint32_t*>(st + C::KC_S + C::KM_S);
      for (int i = lane; i < R * 32; i += 32) kx[i] = 0.f;
      __syncwarp();
      for (int e = lane; e < nout; e += 32) {
        const uint32_t en = ko[e];
        const int pos = static_cast<int>(en >> 16), j = pos / D, c = pos % D;
        const float x = __half2float(__ushort_as_half(static_cast<unsigned short>(en & 0xffffu)));
        const float dz = x - __high2float(km[c]);
#pragma unroll
        for (int r = 0; r < R; ++r) atomicAdd(&kx[r * 32 + j], os[r * D + c] * dz);
      }
      __syncwarp();
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float z = lane_factor(kz, nt);
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        s4[nt][2 * mt] = fmaf(ek2, sc[mt][nt][0] + sc[mt][nt][1], z);
        s4[nt][2 * mt + 1] = fmaf(ek2 * C::RK, sc[mt][nt][2] + sc[mt][nt][3], z);
      }
      if constexpr (OUT) {
        const int r = 4 * nt + t;
        if (r < R) {
#pragma unroll
          for (int k = 0; k < 4; ++k) s4[nt][k] += kx[r * 32 + g + 8 * k];
        }
      }
      if (4 * nt + t < R) {
        const float bm = fmaxf(fmaxf(s4[nt][0], s4[nt][1]), fmaxf(s4[nt][2], s4[nt][3]));
        // vcode_log2(0) is the offset of token g; mlk[nt][0] = m - that
        dmax = fmaxf(dmax, bm - (mlk[nt][0] + static_cast<float>(vcode_log2<BV>(0))));
      }
    }
    if (__any_sync(0xffffffffu, dmax > kLazyMax)) {
      // rare: the pair's first block, or a score far above the maximum
      float mxl[NT], mx[R];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float v = fmaxf(fmaxf(s4[nt][0], s4[nt][1]), fmaxf(s4[nt][2], s4[nt][3]));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
        mxl[nt] = v;
      }
#pragma unroll
      for (int r = 0; r < R; ++r) mx[r] = __shfl_sync(0xffffffffu, mxl[r >> 2], r & 3);
      raise_max(mx);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float pf[4];
      float lp = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        pf[k] = fast_exp2(s4[nt][k] - mlk[nt][k]);
        lp = fmaf(pf[k], pow2i(-vcode_log2<BV>(8 * k)), lp);
      }
      const int r = 4 * nt + t;
      if (r < R) {
        pb[r * 32 + g] = pf[0];
        pb[r * 32 + g + 8] = pf[1];
        pb[r * 32 + g + 16] = pf[2];
        pb[r * 32 + g + 24] = pf[3];
      }
#pragma unroll
      for (int rr = 4 * nt; rr < 4 * nt + 4 && rr < R; ++rr)
        if (t == rr - 4 * nt) lq[rr] += lp;
    }
    __syncwarp();
  };

  // Value operand from the weights in pb (which carry the code factor):
  // items (token pair, group) -> raw pf * s, exponent ev, hi/lo.
  auto v_prep = [&](const uint8_t* st) {
    const __half2* vm = reinterpret_cast<const __half2*>(st + voff + C::VC_S);
    if constexpr (OUT) {
      // kept value outliers: the dense path weighed them as their group's
      // zero point; channel c gains p_j (x - z_jg) for each kept (j, c)
      const uint32_t* vo = reinterpret_cast<const uint32_t*>(st + voff + C::VC_S + C::VM_S);
      for (int e = lane; e < nout; e += 32) {
        const uint32_t en = vo[e];
        const int pos = static_cast<int>(en >> 16), j = pos / D, c = pos % D;
        const float x = __half2float(__ushort_as_half(static_cast<unsigned short>(en & 0xffffu)));
        const float dz = x - __high2float(vm[j * NG + (c >> 5)]);
        const float fj = pow2i(-vcode_log2<BV>(j));
#pragma unroll
        for (int r = 0; r < R; ++r) atomicAdd(&vx[r * D + c], pb[r * 32 + j] * fj * dz);
      }
    }
    float raw[R][VJ][2];
    float vmax = 0.f;
    float2 pp[R];
#pragma unroll
    for (int r = 0; r < R; ++r) pp[r] = *reinterpret_cast<const float2*>(pb + r * 32 + tau0);
#pragma unroll
    for (int i = 0; i < VJ; ++i) {
      const int gp = (lane >> 4) + 2 * i;
      const float2 m0 = __half22float2(vm[tau0 * NG + gp]);
      const float2 m1 = __half22float2(vm[(tau0 + 1) * NG + gp]);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        raw[r][i][0] = pp[r].x * m0.x;
        raw[r][i][1] = pp[r].y * m1.x;
        corr[r][i] = fmaf(pp[r].x, m0.y, fmaf(pp[r].y, m1.y, corr[r][i]));
        vmax = fmaxf(vmax, fmaxf(raw[r][i][0], raw[r][i][1]));
      }
    }
    // B_V = raw * 2^-ev must stay below 2^14; a trip (the first sub-block of a
    // pair, or larger weights/scales later) raises ev and rescales exactly.
    const float va = warp_max_nonneg(vmax);
    if (va * pow2i(min(-ev, 127)) >= 16384.f) {
      const int evn = ilog2f(va) - 13;
      if (evn > ev) {
        const float fv = pow2i(max(ev - evn, -126));
#pragma unroll
        for (int a = 0; a < MTV; ++a)
#pragma unroll
          for (int b = 0; b < NT; ++b)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[a][b][k] *= fv;
        ev = evn;
      }
    }
    const float sv = pow2i(min(-ev, 127));
#pragma unroll
    for (int i = 0; i < VJ; ++i) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float v0 = raw[r][i][0] * sv, v1 = raw[r][i][1] * sv;
        const __half2 hi = __floats2half2_rn(v0, v1);
        const float2 hf = __half22float2(hi);
        const __half2 lo = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
        vb32[vbo[i] + bcol<BSTR>(2 * r)] = *reinterpret_cast<const uint32_t*>(&hi);
        vb32[vbo[i] + bcol<BSTR>(2 * r + 1)] = *reinterpret_cast<const uint32_t*>(&lo);
      }
    }
    __syncwarp();
  };

  auto v_mma = [&](const uint8_t* st) {
    const uint32_t* vc = reinterpret_cast<const uint32_t*>(st + voff);
    // ---- values: O[c][2r+h] += sum_tok A_V[c][tok] * B_V[tok][2r+h]
    if constexpr (BV == 8) {
#pragma unroll
      for (int mt = 0; mt < MTV; ++mt) {
        const int gp = mt >> 1;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          uint32_t a0, a1, a2, a3;
          frag_a8<F8>(words8<2>(vc, mt, ks, lane), a0, a1, a2, a3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint2 b = vbv[((gp * 2 + ks) * NT + nt) * BSTR + blane];
            mma_16816(acc[mt][nt], a0, a1, a2, a3, b.x, b.y);
          }
        }
      }
    } else {
      uint32_t vw[C::VWL];
#pragma unroll
      for (int q = 0; q < C::VWL / 4; ++q) {
        const uint4 x = reinterpret_cast<const uint4*>(vc)[q * 32 + lane];
        vw[4 * q] = x.x; vw[4 * q + 1] = x.y; vw[4 * q + 2] = x.z; vw[4 * q + 3] = x.w;
      }
#pragma unroll
      for (int mt = 0; mt < MTV; ++mt) {
        const int gp = mt >> 1;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          uint32_t a0, a1, a2, a3;
          if constexpr (BV == 2) frag_a2(vw[mt], ks, a0, a1, a2, a3);
          else frag_a4(vw[2 * mt + ks], a0, a1, a2, a3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint2 b = vbv[((gp * 2 + ks) * NT + nt) * BSTR + blane];
            mma_16816(acc[mt][nt], a0, a1, a2, a3, b.x, b.y);
          }
        }
      }
    }
  };

  // Keys stored before RoPE: one 32-token sub-block (sub-block ju of the
  // pair) in stage `st`, scores on CUDA cores (lane = token), then the value
  // operand and mma.
  auto process_sub_rope = [&](const uint8_t* st, int ju) {
    const __half2* km = reinterpret_cast<const __half2*>(st + C::KC_S);
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(st);
    // ---- rotated keys (CUDA cores).  Sub-block positions p0 + j, p0 = 32*ju:
    // q . R(p0 + j) k_j = q' . R(j) k_j with q' = R(-p0) q, and with
    // k = s*c + z per channel, for the pair (i, i+D/2):
    //   cos(j th_i) (al c_i + be c_i2 + ze) + sin(j th_i) (ga c_i + de c_i2 + et).
    // Integer codes are read as x = 1 + c 2^-BK (the code in the mantissa of
    // 1.0, no conversion instruction): the coefficients are scaled by 2^BK
    // and the constant terms absorb the 1s.  Two frequency pairs travel
    // together through packed fp32x2 FMAs.
    constexpr int H = D / 2, F = D / 4;
    constexpr bool MANT = !F8 && BK != 8;
    constexpr float KSC = MANT ? static_cast<float>(1 << BK) : 1.f;
    float* cf = reinterpret_cast<float*>(ws + C::OFF_CF);
    const float2* rrow = reinterpret_cast<const float2*>(st + C::BLK);  // cos/sin(p0 th_i)
    for (int i = lane; i < H; i += 32) {
      const float2 cs = rrow[i];
      const float2 m0 = __half22float2(km[i]), m1 = __half22float2(km[i + H]);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float qi = os[r * D + i], qh = os[r * D + i + H];
        const float ui = fmaf(qi, cs.x, qh * cs.y);   // q'_i
        const float uh = fmaf(qh, cs.x, -qi * cs.y);  // q'_{i+H}
        const float al = ui * m0.x * KSC, be = uh * m1.x * KSC;
        const float ga = uh * m0.x * KSC, de = -ui * m1.x * KSC;
        float ze = fmaf(ui, m0.y, uh * m1.y), et = fmaf(uh, m0.y, -ui * m1.y);
        if constexpr (MANT) {
          ze -= al + be;
          et -= ga + de;
        }
        float* c = cf + (r * F + (i >> 1)) * 12 + (i & 1);
        c[0] = al;
        c[2] = be;
        c[4] = ze;
        c[6] = ga;
        c[8] = de;
        c[10] = et;
      }
    }
    __syncwarp();
    // lane = token: its key codes.  Token 16 mt + 8 hr + g2 sits in lanes
    // 4 g2 + t of the words of m-tile mt (fragment order): 2- and 4-bit
    // words are held in registers, 8-bit codes are read as bytes.
    constexpr int NKR = BK == 8 ? 1 : 4 * (C::KWL / 2);
    uint32_t kr[NKR];
    const int mt = lane >> 4, g2 = lane & 7, hr = (lane >> 3) & 1;
    if constexpr (BK != 8) {
      constexpr int WPM = C::KWL / 2;  // words per m-tile
      // word w of (row g2, slot tq) is component w & 3 of 16-byte chunk
      // (w >> 2) * 32 + 4 g2 + tq: one 16-byte load brings four words
      const uint4* kc4 = reinterpret_cast<const uint4*>(kc);
      if constexpr (WPM >= 4) {
#pragma unroll
        for (int q4 = 0; q4 < WPM / 4; ++q4)
#pragma unroll
          for (int tq = 0; tq < 4; ++tq) {
            const uint4 v = kc4[(mt * (WPM / 4) + q4) * 32 + 4 * g2 + tq];
            kr[(4 * q4 + 0) * 4 + tq] = v.x;
            kr[(4 * q4 + 1) * 4 + tq] = v.y;
            kr[(4 * q4 + 2) * 4 + tq] = v.z;
            kr[(4 * q4 + 3) * 4 + tq] = v.w;
          }
      } else {  // two words per m-tile: both m-tiles share a chunk (w = 2 mt + ww)
#pragma unroll
        for (int tq = 0; tq < 4; ++tq) {
          const uint4 v = kc4[4 * g2 + tq];
          kr[tq] = mt ? v.z : v.x;
          kr[4 + tq] = mt ? v.w : v.y;
        }
      }
    }
    // right rotation that brings the code field of (e, row half hr,
    // pi = 2 (ks % 2) + kh) to the mantissa bits [23 - BK, 23)
    int rot[2][4];
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int pi = 0; pi < 4; ++pi) {
        const int bit = BK == 2 ? 16 * e + (hr ? 2 + 2 * pi : (pi ? 8 + 2 * pi : 0))
                                : 16 * e + 8 * (pi & 1) + 4 * hr;
        rot[e][pi] = (bit - (23 - BK)) & 31;
      }
    // the code of channel d as a float: 1 + c 2^-BK (MANT), else its value
    auto kval = [&](int d) -> float {
      const int ks = d >> 4, kh = (d >> 3) & 1, tq = (d >> 1) & 3, e = d & 1;
      if constexpr (BK == 2) {
        const uint32_t w = kr[(ks >> 1) * 4 + tq];
        return __uint_as_float((__funnelshift_r(w, w, rot[e][2 * (ks & 1) + kh]) & (3u << 21)) |
                               0x3F800000u);
      } else if constexpr (BK == 4) {
        const uint32_t w = kr[ks * 4 + tq];
        return __uint_as_float((__funnelshift_r(w, w, rot[e][kh]) & (15u << 19)) | 0x3F800000u);
      } else {
        const int w = 2 * (mt * KS + ks) + kh;
        const uint8_t* kb = reinterpret_cast<const uint8_t*>(kc);
        return code_value<F8>(kb[(((w >> 2) * 32 + 4 * g2 + tq) * 4 + (w & 3)) * 4 + 2 * hr + e]);
      }
    };
    float2 sc2[R];
#pragma unroll
    for (int r = 0; r < R; ++r) sc2[r] = make_float2(0.f, 0.f);
    const float4* cf4 = reinterpret_cast<const float4*>(cf);
#pragma unroll
    for (int f = 0; f < F; ++f) {
      const float2 x0 = make_float2(kval(2 * f), kval(2 * f + 1));
      const float2 x1 = make_float2(kval(2 * f + H), kval(2 * f + 1 + H));
      const float4 cs = cs_tab[f * 32 + lane];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float4 c0 = cf4[(r * F + f) * 3];      // al, be
        const float4 c1 = cf4[(r * F + f) * 3 + 1];  // ze, ga
        const float4 c2 = cf4[(r * F + f) * 3 + 2];  // de, et
        const float2 A = __ffma2_rn(make_float2(c0.x, c0.y), x0,
                                    __ffma2_rn(make_float2(c0.z, c0.w), x1, make_float2(c1.x, c1.y)));
        const float2 B = __ffma2_rn(make_float2(c1.z, c1.w), x0,
                                    __ffma2_rn(make_float2(c2.x, c2.y), x1, make_float2(c2.z, c2.w)));
        sc2[r] = __ffma2_rn(make_float2(cs.x, cs.y), A, __ffma2_rn(make_float2(cs.z, cs.w), B, sc2[r]));
      }
    }
    float sc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) sc[r] = sc2[r].x + sc2[r].y;
    float mx[R];
#pragma unroll
    for (int r = 0; r < R; ++r) mx[r] = warp_max(sc[r]);
    raise_max(mx);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float pj = fast_exp2(sc[r] - m[r]);
      lq[r] += pj;
      pb[r * 32 + lane] = pj * vfl;
    }
    __syncwarp();
    v_prep(st);
    v_mma(st);
    __syncwarp();
  };

  // fp16 chunk of n <= TCH rows (tail or sink window; its K rows then its V
  // rows in the stage), row j at position pos0 + j.  Lane l holds channels
  // [l*CPL, (l+1)*CPL) (rotated keys: the frequency pairs (i, i + D/2),
  // i = l + 32f); a token's score is the warp sum of the lanes' dot products,
  // JB tokens at a time so that their reductions overlap.  The scaled query
  // sits in `os` (free until the pair's partial is written).
  auto process_chunk = [&](const uint8_t* st, int n, int pos0) {
    const __half* kt = reinterpret_cast<const __half*>(st);
    const __half* vt = kt + TCH * D;
    constexpr int JB = R >= 8 ? 1 : 8 / R;
    if constexpr (ROPE) {
      // key of row j at absolute position pos0 + j, rotated after
      // dequantization: (k_i cos - k_{i+H} sin, k_{i+H} cos + k_i sin)
      constexpr int H = D / 2, FPL = H / 32;
      float qa[R][FPL], qb[R][FPL];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int f = 0; f < FPL; ++f) {
          qa[r][f] = os[r * D + lane + 32 * f];
          qb[r][f] = os[r * D + lane + 32 * f + H];
        }
#pragma unroll
      for (int j0 = 0; j0 < TCH; j0 += JB) {
        float v[JB][R];
#pragma unroll
        for (int jj = 0; jj < JB; ++jj) {
          const int j = j0 + jj;
#pragma unroll
          for (int r = 0; r < R; ++r) v[jj][r] = 0.f;
          if (j < TCH) {
            const float2* cs = p.rope_tab + static_cast<size_t>(pos0 + min(j, n - 1)) * H + lane;
#pragma unroll
            for (int f = 0; f < FPL; ++f) {
              const float2 c = cs[32 * f];
              const float k0 = __half2float(kt[j * D + lane + 32 * f]);
              const float k1 = __half2float(kt[j * D + lane + 32 * f + H]);
              const float r0 = k0 * c.x - k1 * c.y;
              const float r1 = k1 * c.x + k0 * c.y;
#pragma unroll
              for (int r = 0; r < R; ++r) v[jj][r] = fmaf(qa[r][f], r0, fmaf(qb[r][f], r1, v[jj][r]));
            }
          }
        }
#pragma unroll
        for (int jj = 0; jj < JB; ++jj)
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const float sj = warp_sum(v[jj][r]);
            if (lane == j0 + jj) pb[r * 32 + lane] = sj;
          }
      }
    } else {
      float qc[R][CPL];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int c = 0; c < CPL; ++c) qc[r][c] = os[r * D + lane * CPL + c];
#pragma unroll
      for (int j0 = 0; j0 < TCH; j0 += JB) {
        float v[JB][R];
#pragma unroll
        for (int jj = 0; jj < JB; ++jj) {
          const int j = j0 + jj;
#pragma unroll
          for (int r = 0; r < R; ++r) v[jj][r] = 0.f;
          if (j < TCH) {
            float kk[CPL];
            const __half* kr = kt + j * D + lane * CPL;
            if constexpr (CPL == 4) {
              const uint2 x = *reinterpret_cast<const uint2*>(kr);
              const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&x.x));
              const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&x.y));
              kk[0] = a.x; kk[1] = a.y; kk[2] = b.x; kk[3] = b.y;
            } else {
#pragma unroll
              for (int c = 0; c < CPL; ++c) kk[c] = __half2float(kr[c]);
            }
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
              for (int c = 0; c < CPL; ++c) v[jj][r] = fmaf(qc[r][c], kk[c], v[jj][r]);
          }
        }
#pragma unroll
        for (int jj = 0; jj < JB; ++jj)
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const float sj = warp_sum(v[jj][r]);
            if (lane == j0 + jj) pb[r * 32 + lane] = sj;
          }
      }
    }
    __syncwarp();
    // rows >= n hold stale stage bytes: their scores are dropped here
    float sc[R], mx[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      sc[r] = lane < n ? pb[r * 32 + lane] : -INFINITY;
      mx[r] = warp_max(sc[r]);
    }
    raise_max(mx);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float pj = fast_exp2(sc[r] - m[r]);
      lq[r] += pj;
      pb[r * 32 + lane] = pj;
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < TCH; ++j) {
      if (j < n) {
        float vv[CPL];
        const __half* vr = vt + j * D + lane * CPL;
        if constexpr (CPL == 4) {
          const uint2 x = *reinterpret_cast<const uint2*>(vr);
          const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&x.x));
          const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&x.y));
          vv[0] = a.x; vv[1] = a.y; vv[2] = b.x; vv[3] = b.y;
        } else {
#pragma unroll
          for (int c = 0; c < CPL; ++c) vv[c] = __half2float(vr[c]);
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float pj = pb[r * 32 + j];
#pragma unroll
          for (int c = 0; c < CPL; ++c) acct[r][c] = fmaf(pj, vv[c], acct[r][c]);
        }
      }
    }
    __syncwarp();
  };

  // unit j >= nsub of a pair: a chunk of its tail, then of its sink window
  auto process_fp16_unit = [&](const uint8_t* st, int j) {
    const PairLens cl = pair_lens(p, cur);
    const int k = j - cl.nsub;
    if (k < cl.ntu) {
      const int t0 = k * TCH;
      process_chunk(st, min(TCH, cl.Tt - t0), cl.Ts + cl.Tq + t0);
    } else {
      const int t0 = (k - cl.ntu) * TCH;
      process_chunk(st, min(TCH, cl.Ts - t0), t0);
    }
  };

  auto write_partial = [&](int pr) {
    const long long slot = static_cast<long long>(gw) + pr;
    const float e2 = pow2i(ev);
    // zero-point sums: item i of lane L is in group 2 i + (L >> 4); this
    // lane's output channels lie in group go = (lane * CPL) >> 5
    const int go = (lane * CPL) >> 5;
    float ct[R], lsum[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float s0 = corr[r][0] * vfinv;
      float s1 = VJ > 1 ? corr[r][VJ - 1] * vfinv : 0.f;
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) {
        s0 += __shfl_xor_sync(0xffffffffu, s0, o);
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      }
      const float a = __shfl_sync(0xffffffffu, s0, 16 * (go & 1));
      const float b = __shfl_sync(0xffffffffu, s1, 16 * (go & 1));
      ct[r] = go < 2 ? a : b;
      lsum[r] = warp_sum(lq[r]);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int r = 4 * nt + t;
      if (r < R) {
#pragma unroll
        for (int mt = 0; mt < MTV; ++mt) {
          os[r * D + 16 * mt + g] = e2 * (acc[mt][nt][0] + acc[mt][nt][1]);
          os[r * D + 16 * mt + g + 8] = (e2 * C::RV) * (acc[mt][nt][2] + acc[mt][nt][3]);
        }
      }
    }
    __syncwarp();
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (lane == 0) p.part_ml[slot * R + r] = make_float2(m[r], lsum[r]);
      float* o = p.part_o + (slot * R + r) * D + lane * CPL;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        float v = os[r * D + lane * CPL + c] + ct[r] + acct[r][c];
        if constexpr (OUT) v += vx[r * D + lane * CPL + c];
        o[c] = v;
      }
    }
    __syncwarp();
    if (p.fused) {
      // Publish this partial, take a ticket; the pair's last warp merges
      // (it never waits for the others: the ticket tells it they are done).
      __threadfence();
      __syncwarp();
      int w0, w1;
      pair_warps(p.map, pr, &w0, &w1);
      int last = 0;
      if (lane == 0) last = atomicAdd(&p.tickets[pr], 1) == w1 - w0;
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        __threadfence();
        // Lane i weighs partials i and i + 32.  The first eight partial rows
        // are loaded together with the weights (one L2 round trip).
        const int nseg = w1 - w0 + 1;  // <= 64 when fused
        constexpr int RB = 8;
#pragma unroll 1
        for (int r = 0; r < R; ++r) {
          float v[RB][CPL];
#pragma unroll
          for (int u = 0; u < RB; ++u) {
            const long long w = w0 + min(u, nseg - 1);
            const float* src = p.part_o + ((w + pr) * R + r) * D + lane * CPL;
            if constexpr (CPL == 4) {
              const float4 x = __ldcg(reinterpret_cast<const float4*>(src));
              v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
            } else {
#pragma unroll
              for (int c = 0; c < CPL; ++c) v[u][c] = __ldcg(src + c);
            }
          }
          float2 a = make_float2(-INFINITY, 0.f), b = a;
          if (lane < nseg) a = __ldcg(&p.part_ml[(w0 + lane + pr) * R + r]);
          if (lane + 32 < nseg) b = __ldcg(&p.part_ml[(w0 + lane + 32 + pr) * R + r]);
          const float ms = warp_max(fmaxf(a.x, b.x));
          const float mb = ms == -INFINITY ? 0.f : ms;  // every partial empty
          const float fa = fast_exp2(a.x - mb), fb = fast_exp2(b.x - mb);
          const float L = warp_sum(fmaf(fa, a.y, fb * b.y));
          float o[CPL];
#pragma unroll
          for (int c = 0; c < CPL; ++c) o[c] = 0.f;
#pragma unroll
          for (int u = 0; u < RB; ++u) {
            const float f = __shfl_sync(0xffffffffu, fa, u);
            if (u < nseg) {
#pragma unroll
              for (int c = 0; c < CPL; ++c) o[c] = fmaf(f, v[u][c], o[c]);
            }
          }
#pragma unroll 1
          for (int wb = RB; wb < nseg; wb += 8) {
            float x8[8][CPL];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const long long w = w0 + min(wb + u, nseg - 1);
              const float* src = p.part_o + ((w + pr) * R + r) * D + lane * CPL;
#pragma unroll
              for (int c = 0; c < CPL; ++c) x8[u][c] = __ldcg(src + c);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int w = wb + u;
              const float f = __shfl_sync(0xffffffffu, w < 32 ? fa : fb, w & 31);
              if (w < nseg) {
#pragma unroll
                for (int c = 0; c < CPL; ++c) o[c] = fmaf(f, x8[u][c], o[c]);
              }
            }
          }
          const float inv = L > 0.f ? 1.f / L : 0.f;
          float* dst = p.out + (static_cast<long long>(pr) * R + r) * D + lane * CPL;
#pragma unroll
          for (int c = 0; c < CPL; ++c) dst[c] = o[c] * inv;
        }
        if (lane == 0) p.tickets[pr] = 0;
      }
    }
  };

  // ---- main loop: unit n = u - ua sits in stage n % NS, phase (n / NS) & 1
  int pr = static_cast<int>(pair_of_unit(p.map, ua));  // the compute cursor (unit j of pair pr)
  int j = ua - static_cast<int>(first_unit(p.map, pr));
  int cnsub = pair_nsub(p, pr), cupp = pair_upp(p, pr);
  int s = 0;
  uint32_t ph = 0u;
  // the next unit to load goes into `stage` (lane 0 issues the copy)
  auto refill = [&](int stage) {
    if (lu < ub) {
      if (lane == 0) issue(stage);
      advance_load();
    }
  };
  // stage of the previous sub-block when its value mma is still pending
  int pend = -1;
  for (int u = ua; u < ub; ++u) {
    const bool newp = pr != cur;
    if (newp) {
      if constexpr (!ROPE) {
        if (pend >= 0) {
          v_mma(ws + pend * STAGE);
          __syncwarp();
          refill(pend);
          pend = -1;
        }
      }
      if (cur >= 0) write_partial(cur);
    }
    if (!mbar_wait_bounded(&bars[s], ph, p.wait_limit)) {
      // Give up: record the error, wait (bounded) for this warp's copies in
      // flight so no bulk copy lands after the CTA exits, and return.
      if (lane == 0) atomicExch(p.err, kDevErrWait);
      for (int k = u; k < lu; ++k)
        mbar_wait_bounded(&bars[(k - ua) % NS], static_cast<uint32_t>(((k - ua) / NS) & 1));
      return;
    }
    const uint8_t* st = ws + s * STAGE;
    if (newp) {
      cur = pr;
      enter_pair(s);
    }
    if constexpr (ROPE) {
      if (j < cnsub)
        process_sub_rope(st, j);
      else
        process_fp16_unit(st, j);
      refill(s);
    } else {
      if (j < cnsub) {
        // keys of this block, then its key mma beside the value mma of the
        // previous block (independent), then softmax and this block's value
        // operand; its value mma waits for the next iteration
        float kz[R], ek2, sc[2][NT][4];
        k_prep(st, kz, ek2);
        if (pend >= 0) {
          k_mma(st, sc);
          v_mma(ws + pend * STAGE);
          __syncwarp();
          refill(pend);
        } else {
          k_mma(st, sc);
          __syncwarp();
        }
        softmax_scores(st, sc, kz, ek2);
        v_prep(st);
        pend = s;
      } else {
        if (pend >= 0) {
          v_mma(ws + pend * STAGE);
          __syncwarp();
          refill(pend);
          pend = -1;
        }
        process_fp16_unit(st, j);
        refill(s);
      }
    }
    if (++s == NS) {
      s = 0;
      ph ^= 1u;
    }
    if (++j == cupp) {
      j = 0;
      ++pr;
      if (u + 1 < ub) {
        cnsub = pair_nsub(p, pr);
        cupp = pair_upp(p, pr);
      }
    }
  }
  if constexpr (!ROPE) {
    if (pend >= 0) {
      v_mma(ws + pend * STAGE);
      __syncwarp();
    }
  }
  if (cur >= 0) write_partial(cur);
}

template <int D, int BK, int BV, int R, bool ROPE, bool F8 = false, bool OUT = false>
cudaError_t decode_mma_prepare(int* warps_per_sm) {
  using C = MmaCfg<D, BK, BV, R, ROPE, OUT>;
  cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<D, BK, BV, R, ROPE, F8, OUT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  int ctas = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &ctas, decode_mma_kernel<D, BK, BV, R, ROPE, F8, OUT>, C::NW * 32, C::SMEM);
  *warps_per_sm = ctas * C::NW;
  return e;
}

template <int D, int BK, int BV, int R, bool ROPE, bool F8 = false, bool OUT = false>
cudaError_t decode_mma_launch(const DecodeParams& p, cudaStream_t stream) {
  using C = MmaCfg<D, BK, BV, R, ROPE, OUT>;
  // programmatic stream serialization: the grid may start while the previous
  // kernel of the stream finishes; it waits for it before any global access
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.n_warps + C::NW - 1) / C::NW);
  cfg.blockDim = dim3(C::NW * 32);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_mma_kernel<D, BK, BV, R, ROPE, F8, OUT>, p);
}

// Every (bits_k, bits_v) pair of the geometry (G = 32, keys per channel,
// values per token); with `out`, the dense-and-sparse variant (2- and 4-bit
// sides, keys stored after RoPE).
template <int D, int R, bool ROPE>
DecodeOps decode_mma_ops_for(int bk, int bv, bool out) {
  if constexpr (!ROPE) {
    if (out) {
#define KVQ_CASE(BK_, BV_)                                                              \
  if (bk == BK_ && bv == BV_)                                                           \
    return DecodeOps{decode_mma_prepare<D, BK_, BV_, R, false, false, true>,            \
                     decode_mma_launch<D, BK_, BV_, R, false, false, true>};
      KVQ_CASE(2, 2) KVQ_CASE(2, 4) KVQ_CASE(4, 2) KVQ_CASE(4, 4)
#undef KVQ_CASE
      return DecodeOps{nullptr, nullptr};
    }
  }
  if (out) return DecodeOps{nullptr, nullptr};
#define KVQ_CASE(BK_, BV_)                                                              \
  if (bk == BK_ && bv == BV_)                                                           \
    return DecodeOps{decode_mma_prepare<D, BK_, BV_, R, ROPE>,                          \
                     decode_mma_launch<D, BK_, BV_, R, ROPE>};
  KVQ_CASE(2, 2) KVQ_CASE(2, 4) KVQ_CASE(2, 8)
  KVQ_CASE(4, 2) KVQ_CASE(4, 4) KVQ_CASE(4, 8)
  KVQ_CASE(8, 2) KVQ_CASE(8, 4) KVQ_CASE(8, 8)
#undef KVQ_CASE
  if (bk == kBitsE4M3 && bv == kBitsE4M3)
    return DecodeOps{decode_mma_prepare<D, 8, 8, R, ROPE, true>,
                     decode_mma_launch<D, 8, 8, R, ROPE, true>};
  return DecodeOps{nullptr, nullptr};
}

// Dispatch over the per-(D, R) translation units (kvq_merge.cu);
// {nullptr, nullptr} when no tensor-core instantiation exists.
DecodeOps decode_mma_ops(int D, int R, int bk, int bv, bool rope, bool out = false);

}  // namespace kvq
