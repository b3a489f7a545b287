// kvq_decode_mma.cuh — tensor-core decode attention for the pages' geometry:
// keys grouped per channel, values grouped per token, G = 32 (the
// configuration "Your KV cache doesn't have a bit problem, it has a geometry
// problem" recommends, section "What to Do with This").
//
// Work split, partials, merge and fp16 tail are those of decode_split_kernel
// (kvq_decode.cuh).  With G = 32 a sub-block is a whole block, so one bulk
// copy of block_bytes moves a unit into a stage; tail units stream their fp16
// rows through the same stages (mma_tail_chunk tokens per unit).
//
// Scores and value sums run on mma.sync with the packed codes themselves as
// one exact operand:
//
//   fp8 path (2- and 4-bit codes, fragment order).  An e4m3 byte n < 16 is
//     exactly n * 2^-9 (subnormals 0..7, then exponent 1), so a code masked
//     in place is an exact operand: one AND gives four codes.  A 2-bit code at
//     bits 2-3 of its byte counts 4x; its k-slots get a 4x smaller other
//     operand.  The other operand (q_d * s_d for scores, p_j * s_j for values)
//     is a fixed-point integer y < 2^23 split into six 4-bit digits, digit i
//     in column i of the 8-column tile (e4m3 byte 0..15, sign in bit 7 for the
//     query side).  Every product is an integer times 2^-18 and every tile sum
//     stays far below 2^24 * 2^-18, so the mma sums are exact; column i is
//     weighted by 16^i when the digits are recombined.
//       scores  m16n8k32: rows = 32 tokens (2 m-tiles), k = 32 channels per
//               slice, one n-tile of six digit columns per query head;
//       values  m16n8k32: rows = D channels, k = the 32 tokens, columns = the
//               six digits (one query head).
//   fp16 path (8-bit codes, and values of 2/4-bit codes with several query
//     heads).  Codes become fp16 registers with masks (8-bit: byte permute to
//     1024 + c minus 1024; 2/4-bit fragment words: 1 + c/16 or 1 + c/4 in the
//     mantissa); the other operand is an fp32 value split into fp16 hi + lo
//     columns (~22 bits), and exact corrections remove the constant 1.
//
// Scores are in log2 units (the query carries scale * log2 e).
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

// e4m3 x e4m3 -> fp32, m16n8k32: a0 = (row g, k 4t..4t+3), a1 = (row g+8, same
// k), a2 = (row g, k 16+4t..), a3 = (row g+8, k 16+4t..); b0 = (k 4t.., col g),
// b1 = (k 16+4t.., col g); d = rows g / g+8 x columns 2t, 2t+1.
__device__ __forceinline__ void mma_f8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                       uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
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

// Byte transpose of four values: T[b] holds byte b of y[0..3] in its bytes
// 0..3 (b < 3).
__device__ __forceinline__ void transpose3(const uint32_t (&y)[4], uint32_t (&T)[3]) {
  const uint32_t a = __byte_perm(y[0], y[1], 0x5140), b = __byte_perm(y[2], y[3], 0x5140);
  T[0] = __byte_perm(a, b, 0x5410);
  T[1] = __byte_perm(a, b, 0x7632);
  T[2] = __byte_perm(__byte_perm(y[0], y[1], 0x0062), __byte_perm(y[2], y[3], 0x0062), 0x5410);
}

// 0x80 in byte j where x[j] is negative.
__device__ __forceinline__ uint32_t sign_bytes(const float (&x)[4]) {
  const uint32_t s01 = __byte_perm(__float_as_uint(x[0]), __float_as_uint(x[1]), 0x00FB);
  const uint32_t s23 = __byte_perm(__float_as_uint(x[2]), __float_as_uint(x[3]), 0x00FB);
  return __byte_perm(s01, s23, 0x5410) & 0x80808080u;
}

// Digit i (4 bits, i < 6) of the four values transposed in T, one per byte.
__device__ __forceinline__ uint32_t digit4(const uint32_t (&T)[3], int i) {
  return ((i & 1) ? (T[i >> 1] >> 4) : T[i >> 1]) & 0x0F0F0F0Fu;
}

// Entry s (of n) of a lane's row of n uint2: rows of four entries are read as
// two 16-byte halves, swapped on every other group of four lanes so that
// eight consecutive lanes cover all 32 banks.
__device__ __forceinline__ int swz(int lane, int s, int n) {
  return n == 4 ? (s ^ (((lane >> 2) & 1) << 1)) : s;
}

// 8-bit codes in sequential order -> fp16 operand registers of one
// 16-element slice: a byte permute builds 1024 + c and one half2 subtraction
// of 1024 leaves the exact code.  x0 covers fragment columns (2t, 2t+1), x2
// covers (2t+8, 2t+9); element e sits in lane lane_t(e), register reg(e).
struct Frag8 {
  static constexpr int PARTNER = 1;  // element sharing lane and register, other half
  __device__ static __forceinline__ int base(int i) { return 2 * i; }
  __device__ static __forceinline__ void get(const uint32_t* w, int t, uint32_t& x0, uint32_t& x2) {
    const uint32_t v = w[t];
    const __half2 k1024 = __float2half2_rn(1024.0f);
    uint32_t p0 = __byte_perm(v, 0x64646464u, 0x4140u);  // 1024 + byte0, 1024 + byte1
    uint32_t p2 = __byte_perm(v, 0x64646464u, 0x4342u);  // 1024 + byte2, 1024 + byte3
    __half2 h0 = __hsub2(*reinterpret_cast<__half2*>(&p0), k1024);
    __half2 h2 = __hsub2(*reinterpret_cast<__half2*>(&p2), k1024);
    x0 = *reinterpret_cast<uint32_t*>(&h0);  // elements 4t, 4t+1 (exact codes)
    x2 = *reinterpret_cast<uint32_t*>(&h2);  // elements 4t+2, 4t+3
  }
  __device__ static __forceinline__ int lane_t(int e) { return e >> 2; }
  __device__ static __forceinline__ int reg(int e) { return (e & 3) >= 2 ? 1 : 0; }
};

template <int D, int BK, int BV, int R, bool ROPE>
struct MmaCfg {
  static constexpr int G = 32;
  static constexpr int NSL = D / 32;              // 32-channel key slices
  static constexpr int NG = D / 32;               // value channel groups
  static constexpr int MTV = D / 16;              // value m-tiles
  static constexpr int CPL = D / 32;              // output channels per lane
  static constexpr bool KF8 = BK <= 4 && !ROPE;   // scores on the fp8 path
  static constexpr bool KFRAG = BK <= 4;          // key codes in fragment order
  static constexpr bool VF8 = BV <= 4 && R == 1;  // values on the fp8 path
  static constexpr bool VFRAG = BV <= 4;          // value codes in fragment order
  static constexpr int NT = (2 * R + 7) / 8;      // fp16 n-tiles = query groups of 4
  static constexpr int NTA = VF8 ? 1 : NT;        // value accumulator n-tiles
  static constexpr int KS = D / 16;               // fp16 key k-steps
  static constexpr int KWL = D * BK / 32;         // key words per lane / per row
  static constexpr int VWL = D * BV / 32;         // value words per lane (fragment)
  static constexpr int KC_S = 4 * D * BK;
  static constexpr int KM_S = 4 * D;
  static constexpr int VC_S = 4 * D * BV;
  static constexpr int VM_S = 4 * D;
  static constexpr int STAGE = KC_S + KM_S + VC_S + VM_S;  // one block
  static constexpr int NS = ROPE ? 2 : (STAGE <= 4096 ? 3 : 2);
  static constexpr int TCH = mma_tail_chunk(BK, BV);
  static constexpr int OFF_BAR = NS * STAGE;
  static constexpr int OFF_KB = OFF_BAR + 64;
  // key operand: fp8 [R][32 lanes][NSL] uint2; fp16 [KS][NT][32] uint2
  static constexpr int KB_BYTES = KF8 ? R * 32 * NSL * 8 : (ROPE ? 0 : KS * NT * 32 * 8);
  static constexpr int OFF_VB = OFF_KB + KB_BYTES;
  // value operand: fp8 [32 lanes][NG] uint2; fp16 [NG][2][NT][32] uint2
  static constexpr int VB_BYTES = VF8 ? 32 * NG * 8 : NG * 2 * NT * 32 * 8;
  static constexpr int OFF_PB = OFF_VB + VB_BYTES;   // [R][32] float
  static constexpr int OFF_OS = OFF_PB + R * 32 * 4; // [R][D] float
  // RoPE: per-warp key coefficients [R][D/2][8] floats; per-CTA table of
  // cos/sin(j * theta_i), j < 32, stored [D/2][32] float2.
  static constexpr int OFF_CF = OFF_OS + R * D * 4;
  static constexpr int WARP_BYTES = round_up(OFF_CF + (ROPE ? R * (D / 2) * 32 : 0), 128);
  static constexpr int CS_BYTES = ROPE ? (D / 2) * 32 * 8 : 0;
  static constexpr int SMEM = kDecodeWarps * WARP_BYTES + CS_BYTES;
  static_assert(2 * TCH * D * 2 == STAGE, "a tail chunk fills one stage");
  static_assert(!KFRAG || KWL % 4 == 0, "lane words are read as 16-byte vectors");
  static_assert(!VFRAG || VWL % 4 == 0, "lane words are read as 16-byte vectors");
};

template <int D, int BK, int BV, int R, bool ROPE>
__global__ void __launch_bounds__(kDecodeWarps * 32, R == 1 ? (ROPE ? 3 : 4) : (R <= 4 ? 3 : 1))
    decode_mma_kernel(const DecodeParams p) {
  using C = MmaCfg<D, BK, BV, R, ROPE>;
  constexpr int NS = C::NS, NT = C::NT, NTA = C::NTA, NSL = C::NSL, NG = C::NG, MTV = C::MTV,
                CPL = C::CPL, TCH = C::TCH, STAGE = C::STAGE, KS = C::KS;

  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const long long gw = static_cast<long long>(blockIdx.x) * kDecodeWarps + warp;
  // RoPE: cos/sin(j * theta_i) for the 32 token offsets of a sub-block (table
  // rows 0..31), transposed so lane j reads its own column conflict-free.
  // Loaded before any warp of the CTA can leave.
  float2* cs_tab = reinterpret_cast<float2*>(smem + kDecodeWarps * C::WARP_BYTES);
  if constexpr (ROPE) {
    for (int idx = threadIdx.x; idx < (D / 2) * 32; idx += blockDim.x) {
      const int i = idx >> 5, j = idx & 31;
      cs_tab[idx] = j < p.rope_rows ? p.rope_tab[static_cast<size_t>(j) * (D / 2) + i]
                                    : make_float2(1.f, 0.f);
    }
    __syncthreads();
  }
  if (gw >= p.n_warps) return;

  uint8_t* ws = smem + warp * C::WARP_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ws + C::OFF_BAR);
  uint32_t* kb32 = reinterpret_cast<uint32_t*>(ws + C::OFF_KB);
  uint32_t* vb32 = reinterpret_cast<uint32_t*>(ws + C::OFF_VB);
  const uint2* kbv = reinterpret_cast<const uint2*>(ws + C::OFF_KB);
  const uint2* vbv = reinterpret_cast<const uint2*>(ws + C::OFF_VB);
  float* pb = reinterpret_cast<float*>(ws + C::OFF_PB);
  float* os = reinterpret_cast<float*>(ws + C::OFF_OS);

  // Operand buffers: entries never written (digit columns 6 and 7, fp16
  // columns >= 2R) stay zero.
  for (int i = lane; i < (C::OFF_PB - C::OFF_KB) / 4; i += 32) kb32[i] = 0u;
  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  // ---- this warp's units [ua, ub) and the load cursor, NS units ahead
  const int ua = static_cast<int>(gw * p.U / p.n_warps);
  const int ub = static_cast<int>((gw + 1) * p.U / p.n_warps);
  const int upp = p.upp, nsub = p.nsub;
  int lu = ua, lpr = ua / upp;
  int lj = ua - lpr * upp;
  const uint8_t* lbase = p.g.blocks + static_cast<size_t>(lpr) * p.g.NB * STAGE;
  auto issue = [&](int s) {  // lane 0: unit (lpr, lj) -> stage s
    uint8_t* st = ws + s * STAGE;
    if (lj < nsub) {
      mbar_arrive_expect_tx(&bars[s], STAGE);
      bulk_g2s(st, lbase + static_cast<size_t>(lj) * STAGE, STAGE, &bars[s]);
    } else {
      const int t0 = (lj - nsub) * TCH;
      const uint32_t bytes = static_cast<uint32_t>(min(TCH, p.T_t - t0)) * D * 2;
      const size_t row = static_cast<size_t>(lpr) * C::G + t0;
      mbar_arrive_expect_tx(&bars[s], 2 * bytes);
      bulk_g2s(st, p.ktail + row * D, bytes, &bars[s]);
      bulk_g2s(st + TCH * D * 2, p.vtail + row * D, bytes, &bars[s]);
    }
  };
  auto advance_load = [&]() {
    ++lu;
    if (++lj == upp) {
      lj = 0;
      ++lpr;
      lbase += static_cast<size_t>(p.g.NB) * STAGE;
    }
  };
  for (int s = 0; s < NS && lu < ub; ++s) {
    if (lane == 0) issue(s);
    advance_load();
  }

  // ---- key items of this lane on the fp8 path: channel quad kQ = channels
  // 32*ksl + 16*khc + 4*kt + {0..3}, for query heads (lane + 32 i) / NQ.
  constexpr int NQ = D / 4;
  constexpr int IPL = (NQ * R + 31) / 32;
  const int kQ = lane % NQ;
  const int ksl = kQ >> 3, khc = (kQ >> 2) & 1, kt = kQ & 3;
  const int kch0 = 32 * ksl + 16 * khc + 4 * kt;
  // channel pairs of this lane on the fp16 key path (8-bit codes)
  constexpr int KP = D / 64;
  auto kchan = [&](int i, int h) {
    const int P = lane + 32 * i;
    return 16 * (P >> 3) + Frag8::base(P & 7) + h * Frag8::PARTNER;
  };
  constexpr int VJ = 2;  // value items per lane on the fp16 path

  float qk[IPL][4];      // fp8 key items: q * scale * log2(e)
  float qreg[R][KP][2];  // fp16 key path: the same
  float m[R], l[R];      // online softmax, identical in all lanes
  float acc[MTV][NTA][4];
  float corr[R][VJ];     // value zero-point sums of this lane's items
  float acct[R][CPL];    // fp16-tail contributions, channels lane*CPL + c
  int ev = -126;         // value operand exponent
  int cur = -1;

  auto enter_pair = [&](int pr) {
    const __half* qp = p.q + static_cast<size_t>(pr) * R * D;
    if constexpr (C::KF8) {
#pragma unroll
      for (int i = 0; i < IPL; ++i) {
        const int r = (lane + 32 * i) / NQ;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          qk[i][j] = r < R ? __half2float(qp[r * D + kch0 + j]) * p.qscale : 0.f;
      }
    } else if constexpr (!ROPE) {
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int i = 0; i < KP; ++i)
#pragma unroll
          for (int h = 0; h < 2; ++h)
            qreg[r][i][h] = __half2float(qp[r * D + kchan(i, h)]) * p.qscale;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      m[r] = -INFINITY;
      l[r] = 0.f;
#pragma unroll
      for (int k = 0; k < VJ; ++k) corr[r][k] = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) acct[r][c] = 0.f;
    }
#pragma unroll
    for (int a = 0; a < MTV; ++a)
#pragma unroll
      for (int b = 0; b < NTA; ++b)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[a][b][k] = 0.f;
    ev = -126;
    // the scaled query, all channels (rotated-key sub-blocks and the tail)
    for (int i = lane; i < R * D; i += 32) os[i] = __half2float(qp[i]) * p.qscale;
    __syncwarp();
  };

  // value of f for this lane's query column (query 4*nt + t), 1 if none
  auto lane_factor = [&](const float (&f)[R], int nt) -> float {
    float v = 1.f;
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (r == 4 * nt + t) v = f[r];
    return v;
  };

  // Multiplies the value accumulators and corrections by per-query factors.
  auto rescale = [&](const float (&f)[R], float fv) {
    bool any = fv != 1.f;
#pragma unroll
    for (int r = 0; r < R; ++r) any |= f[r] != 1.f;
    if (!any) return;  // warp-uniform
#pragma unroll
    for (int nt = 0; nt < NTA; ++nt) {
      const float lf = (C::VF8 ? f[0] : lane_factor(f, nt)) * fv;
#pragma unroll
      for (int a = 0; a < MTV; ++a)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[a][nt][k] *= lf;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
      for (int k = 0; k < VJ; ++k) corr[r][k] *= f[r];
#pragma unroll
      for (int c = 0; c < CPL; ++c) acct[r][c] *= f[r];
    }
  };

  auto softmax_merge = [&](const float (&mx)[R], float (&alpha)[R], float (&mnew)[R]) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      mnew[r] = fmaxf(m[r], mx[r]);
      alpha[r] = fast_exp2(m[r] - mnew[r]);
      m[r] = mnew[r];
    }
  };

  // One 32-token sub-block (sub-block ju of the pair) in stage `st`.
  auto process_sub = [&](const uint8_t* st, int ju) {
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(st);
    const __half2* km = reinterpret_cast<const __half2*>(st + C::KC_S);
    const uint32_t* vc = reinterpret_cast<const uint32_t*>(st + C::KC_S + C::KM_S);
    const __half2* vm = reinterpret_cast<const __half2*>(st + C::KC_S + C::KM_S + C::VC_S);

    float alpha[R];
    if constexpr (ROPE) {
      // ---- rotated keys (CUDA cores).  Sub-block positions p0 + j, p0 = 32*ju:
      // q . R(p0 + j) k_j = q' . R(j) k_j with q' = R(-p0) q, and with
      // k = s*c + z per channel, for the pair (i, i+D/2):
      //   cos(j th_i) (a c_i + b c_i2 + e) + sin(j th_i) (f c_i - g c_i2 + h).
      constexpr int H = D / 2;
      float* cf = reinterpret_cast<float*>(ws + C::OFF_CF);
      const int p0 = ju * 32;
      for (int i = lane; i < H; i += 32) {
        const float2 cs = p.rope_tab[static_cast<size_t>(p0) * H + i];
        const float2 m0 = __half22float2(km[i]), m1 = __half22float2(km[i + H]);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float qi = os[r * D + i], qh = os[r * D + i + H];
          const float ui = fmaf(qi, cs.x, qh * cs.y);   // q'_i
          const float uh = fmaf(qh, cs.x, -qi * cs.y);  // q'_{i+H}
          float* c = cf + (r * H + i) * 8;
          *reinterpret_cast<float4*>(c) =
              make_float4(ui * m0.x, uh * m1.x, fmaf(ui, m0.y, uh * m1.y), uh * m0.x);
          *reinterpret_cast<float2*>(c + 4) = make_float2(ui * m1.x, fmaf(uh, m0.y, -ui * m1.y));
        }
      }
      __syncwarp();
      // lane = token: its key codes.  Fragment order: token = 16 mt + 8 hr + g2
      // sits in lanes 4 g2 + tq of words mt*NSL + s (2-bit) or 2(mt*NSL + s) + hc
      // (4-bit), shifted by 4 hr; sequential order: one row of KWL words.
      constexpr int NKR = C::KFRAG ? NSL * 4 * (BK / 2) : C::KWL;
      uint32_t kr[NKR];
      if constexpr (C::KFRAG) {
        const int mt = lane >> 4, hr = (lane >> 3) & 1, g2 = lane & 7;
#pragma unroll
        for (int s = 0; s < NSL; ++s)
#pragma unroll
          for (int tq = 0; tq < 4; ++tq)
#pragma unroll
            for (int h = 0; h < BK / 2; ++h) {
              const int w = BK == 2 ? mt * NSL + s : 2 * (mt * NSL + s) + h;
              kr[(s * 4 + tq) * (BK / 2) + h] = kc[((w >> 2) * 32 + 4 * g2 + tq) * 4 + (w & 3)] >> (4 * hr);
            }
      } else {
        const uint4* row = reinterpret_cast<const uint4*>(kc + lane * C::KWL);
#pragma unroll
        for (int v = 0; v < C::KWL / 4; ++v) {
          const uint4 w4 = row[v];
          kr[4 * v] = w4.x; kr[4 * v + 1] = w4.y; kr[4 * v + 2] = w4.z; kr[4 * v + 3] = w4.w;
        }
      }
      auto kcode = [&](int d) -> uint32_t {
        if constexpr (C::KFRAG) {
          const int s = d >> 5, hc = (d >> 4) & 1, tq = (d >> 2) & 3, j = d & 3;
          if constexpr (BK == 2) return (kr[s * 4 + tq] >> (8 * j + 2 * hc)) & 3u;
          else return (kr[(s * 4 + tq) * 2 + hc] >> (8 * j)) & 15u;
        } else {
          constexpr int KPER = 32 / BK;
          return (kr[d / KPER] >> ((d % KPER) * BK)) & ((1u << BK) - 1u);
        }
      };
      float sc[R];
#pragma unroll
      for (int r = 0; r < R; ++r) sc[r] = 0.f;
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const float c0 = code_to_float(kcode(i));
        const float c1 = code_to_float(kcode(i + H));
        const float2 cs = cs_tab[i * 32 + lane];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float4 ab = *reinterpret_cast<const float4*>(cf + (r * H + i) * 8);
          const float2 gh = *reinterpret_cast<const float2*>(cf + (r * H + i) * 8 + 4);
          const float A = fmaf(ab.x, c0, fmaf(ab.y, c1, ab.z));
          const float B = fmaf(ab.w, c0, fmaf(-gh.x, c1, gh.y));
          sc[r] = fmaf(cs.x, A, fmaf(cs.y, B, sc[r]));
        }
      }
      float mx[R], mnew[R];
#pragma unroll
      for (int r = 0; r < R; ++r) mx[r] = warp_max(sc[r]);
      softmax_merge(mx, alpha, mnew);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float pj = fast_exp2(sc[r] - mnew[r]);
        l[r] = l[r] * alpha[r] + warp_sum(pj);
        pb[r * 32 + lane] = pj;
      }
      __syncwarp();
    } else {
      // ---- scores -> s4[nt][k]: query 4*nt + t, token 8*k + g
      float s4[NT][4];
      if constexpr (C::KF8) {
        // key operand: X = q_d * s_d as y = rint(|X| 2^F) (4 y for the k-slots
        // whose codes count 4x), six 4-bit digits per value
        const uint4 m4 = *reinterpret_cast<const uint4*>(km + kch0);
        const uint32_t mw[4] = {m4.x, m4.y, m4.z, m4.w};
        float2 sz[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) sz[j] = __half22float2(*reinterpret_cast<const __half2*>(&mw[j]));
        float kzp[IPL];
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < IPL; ++i) {
          kzp[i] = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            kzp[i] = fmaf(qk[i][j], sz[j].y, kzp[i]);
            amax = fmaxf(amax, fabsf(qk[i][j] * sz[j].x));
          }
        }
        amax = warp_max(amax);
        const int F = min((BK == 2 ? 19 : 21) - ilog2f(amax), 120);
        const float mult = pow2i((BK == 2 && khc == 0) ? F + 2 : F);
#pragma unroll
        for (int i = 0; i < IPL; ++i) {
          const int r = (lane + 32 * i) / NQ;
          if (r < R) {
            float X[4];
            uint32_t y[4], T[3];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              X[j] = qk[i][j] * sz[j].x;
              y[j] = __float2uint_rn(fabsf(X[j]) * mult);
            }
            const uint32_t S = sign_bytes(X);
            transpose3(y, T);
#pragma unroll
            for (int dg = 0; dg < 6; ++dg) {
              const int ln = 4 * dg + kt;
              kb32[((r * 32 + ln) * NSL + swz(ln, ksl, NSL)) * 2 + khc] = digit4(T, dg) | S;
            }
          }
        }
        // zero-point term per query: sum over the lanes holding that query
        float kz[R];
        if constexpr (NQ == 32) {
#pragma unroll
          for (int r = 0; r < R; ++r) kz[r] = warp_sum(kzp[r]);
        } else {
          float kh[IPL];
#pragma unroll
          for (int i = 0; i < IPL; ++i) {
            float v = kzp[i];
#pragma unroll
            for (int o = 1; o < NQ; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            kh[i] = v;  // query (lane + 32 i) / NQ
          }
#pragma unroll
          for (int r = 0; r < R; ++r)
            kz[r] = __shfl_sync(0xffffffffu, kh[(r * NQ) / 32], (r * NQ) % 32);
        }
        __syncwarp();
        // scores: A = this lane's key words, B = the digit columns of query r
        uint32_t kw[C::KWL];
#pragma unroll
        for (int q = 0; q < C::KWL / 4; ++q) {
          const uint4 x = reinterpret_cast<const uint4*>(kc)[q * 32 + lane];
          kw[4 * q] = x.x; kw[4 * q + 1] = x.y; kw[4 * q + 2] = x.z; kw[4 * q + 3] = x.w;
        }
        float sc[2][R][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int r = 0; r < R; ++r)
#pragma unroll
            for (int k = 0; k < 4; ++k) sc[mt][r][k] = 0.f;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int s = 0; s < NSL; ++s) {
            uint32_t a0, a1, a2, a3;
            if constexpr (BK == 2) {
              const uint32_t w = kw[mt * NSL + s], x = w >> 4;
              a0 = w & 0x03030303u; a2 = w & 0x0C0C0C0Cu;
              a1 = x & 0x03030303u; a3 = x & 0x0C0C0C0Cu;
            } else {
              const uint32_t w0 = kw[2 * (mt * NSL + s)], w1 = kw[2 * (mt * NSL + s) + 1];
              a0 = w0 & 0x0F0F0F0Fu; a1 = (w0 >> 4) & 0x0F0F0F0Fu;
              a2 = w1 & 0x0F0F0F0Fu; a3 = (w1 >> 4) & 0x0F0F0F0Fu;
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
              const uint2 b = kbv[(r * 32 + lane) * NSL + swz(lane, s, NSL)];
              mma_f8(sc[mt][r], a0, a1, a2, a3, b.x, b.y);
            }
          }
        // digits 2t, 2t+1 of this lane -> value; sum over the quad
        const float f0 = pow2i(8 * t), f1 = pow2i(8 * t + 4);
        const float ss = pow2i((BK == 2 ? 16 : 18) - F);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            float v[R];
#pragma unroll
            for (int r = 0; r < R; ++r) v[r] = fmaf(sc[mt][r][2 * hr], f0, sc[mt][r][2 * hr + 1] * f1);
            if constexpr (R <= 2) {
#pragma unroll
              for (int r = 0; r < R; ++r) {
                v[r] += __shfl_xor_sync(0xffffffffu, v[r], 1);
                v[r] += __shfl_xor_sync(0xffffffffu, v[r], 2);
              }
              const float vq = (R == 2 && (t & 1)) ? v[R - 1] : v[0];
              const float zq = (R == 2 && (t & 1)) ? kz[R - 1] : kz[0];
              s4[0][2 * mt + hr] = fmaf(vq, ss, zq);
            } else {
              // reduce-scatter over the quad: lane t keeps query 4*nt + t
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                const bool b0 = t & 1, b1 = (t >> 1) & 1;
                float k0 = b0 ? v[4 * nt + 1] : v[4 * nt], s0 = b0 ? v[4 * nt] : v[4 * nt + 1];
                float k1 = b0 ? v[4 * nt + 3] : v[4 * nt + 2], s1 = b0 ? v[4 * nt + 2] : v[4 * nt + 3];
                k0 += __shfl_xor_sync(0xffffffffu, s0, 1);
                k1 += __shfl_xor_sync(0xffffffffu, s1, 1);
                float kk = b1 ? k1 : k0;
                kk += __shfl_xor_sync(0xffffffffu, b1 ? k0 : k1, 2);
                s4[nt][2 * mt + hr] = fmaf(kk, ss, lane_factor(kz, nt));
              }
            }
          }
      } else {
        // ---- fp16 key path (8-bit codes): B_K[c][2r+h] = hi/lo of q_r[c] s_c 2^-ek
        float qh[R][KP][2];
        float kz[R];
        float amax = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) kz[r] = 0.f;
#pragma unroll
        for (int i = 0; i < KP; ++i) {
          const float2 s0 = __half22float2(km[kchan(i, 0)]);
          const float2 s1 = __half22float2(km[kchan(i, 1)]);
#pragma unroll
          for (int r = 0; r < R; ++r) {
            qh[r][i][0] = qreg[r][i][0] * s0.x;
            qh[r][i][1] = qreg[r][i][1] * s1.x;
            kz[r] = fmaf(qreg[r][i][0], s0.y, fmaf(qreg[r][i][1], s1.y, kz[r]));
            amax = fmaxf(amax, fmaxf(fabsf(qh[r][i][0]), fabsf(qh[r][i][1])));
          }
        }
        amax = warp_max(amax);
        const int ek = max(0, ilog2f(amax) - 13);
        const float sk = pow2i(-ek), ek2 = pow2i(ek);
#pragma unroll
        for (int i = 0; i < KP; ++i) {
          const int P = lane + 32 * i;
          const int kk = P >> 3, e0 = Frag8::base(P & 7);
          const int slot_t = Frag8::lane_t(e0), rg = Frag8::reg(e0);
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const float v0 = qh[r][i][0] * sk, v1 = qh[r][i][1] * sk;
            const __half2 hi = __floats2half2_rn(v0, v1);
            const float2 hf = __half22float2(hi);
            const __half2 lo = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
            const int n0 = 2 * r, n1 = 2 * r + 1;
            kb32[((kk * NT + (n0 >> 3)) * 32 + (n0 & 7) * 4 + slot_t) * 2 + rg] =
                *reinterpret_cast<const uint32_t*>(&hi);
            kb32[((kk * NT + (n1 >> 3)) * 32 + (n1 & 7) * 4 + slot_t) * 2 + rg] =
                *reinterpret_cast<const uint32_t*>(&lo);
          }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) kz[r] = warp_sum(kz[r]);
        __syncwarp();
        float sc[2][NT][4];
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int b = 0; b < NT; ++b)
#pragma unroll
            for (int k = 0; k < 4; ++k) sc[a][b][k] = 0.f;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const uint32_t* r0 = kc + (16 * mt + g) * C::KWL;
          const uint32_t* r1 = r0 + 8 * C::KWL;
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            uint32_t a0, a1, a2, a3;
            Frag8::get(r0 + kk * 4, t, a0, a2);
            Frag8::get(r1 + kk * 4, t, a1, a3);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const uint2 b = kbv[(kk * NT + nt) * 32 + lane];
              mma_16816(sc[mt][nt], a0, a1, a2, a3, b.x, b.y);
            }
          }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float z = lane_factor(kz, nt);
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            s4[nt][2 * mt] = fmaf(ek2, sc[mt][nt][0] + sc[mt][nt][1], z);
            s4[nt][2 * mt + 1] = fmaf(ek2, sc[mt][nt][2] + sc[mt][nt][3], z);
          }
        }
      }

      // ---- online softmax (log2 units); lane holds query 4*nt + t
      float mx[R], mxl[NT];
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
      float mnew[R];
      softmax_merge(mx, alpha, mnew);
      float ps[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float mm = lane_factor(mnew, nt);
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          s4[nt][k] = fast_exp2(s4[nt][k] - mm);
          sum += s4[nt][k];
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        sum += __shfl_xor_sync(0xffffffffu, sum, 8);
        sum += __shfl_xor_sync(0xffffffffu, sum, 16);
        ps[nt] = sum;
        const int r = 4 * nt + t;
        if (r < R) {
          pb[r * 32 + g] = s4[nt][0];
          pb[r * 32 + g + 8] = s4[nt][1];
          pb[r * 32 + g + 16] = s4[nt][2];
          pb[r * 32 + g + 24] = s4[nt][3];
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r)
        l[r] = l[r] * alpha[r] + __shfl_sync(0xffffffffu, ps[r >> 2], r & 3);
      __syncwarp();
    }

    // ---- values
    if constexpr (C::VF8) {
      // value operand: W = p_j * s_j as y = rint(W 2^-ev) (4 y for the tokens
      // whose codes count 4x), six digits.  Item of this lane: group vgp,
      // tokens 16*vhc + 4*vt + {0..3}.
      const int vgp = lane >> 3, vhc = (lane >> 2) & 1, vt = lane & 3;
      const bool vvalid = vgp < NG;
      const int tau0 = 16 * vhc + 4 * vt;
      const float4 p4 = *reinterpret_cast<const float4*>(pb + tau0);
      const float pv[4] = {p4.x, p4.y, p4.z, p4.w};
      float W[4], zz = 0.f, vmax = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 sz = vvalid ? __half22float2(vm[(tau0 + j) * NG + vgp]) : make_float2(0.f, 0.f);
        W[j] = pv[j] * sz.x;
        zz = fmaf(pv[j], sz.y, zz);
        vmax = fmaxf(vmax, W[j]);
      }
      // y must stay below 2^22: W 2^-ev < 2^20 (2-bit) / 2^22 (4-bit); a trip
      // raises ev and rescales the accumulators exactly
      constexpr float VLIM = BV == 2 ? 1048576.f : 4194304.f;
      float fv = 1.f;
      if (__any_sync(0xffffffffu, vmax * pow2i(-ev) >= VLIM)) {
        const float va = warp_max(vmax);
        const int evn = ilog2f(va) - (BV == 2 ? 19 : 21);
        if (evn > ev) {
          fv = pow2i(max(ev - evn, -126));
          ev = evn;
        }
      }
      rescale(alpha, fv);
      corr[0][0] += zz;
      const float mult = pow2i(min(127, ((BV == 2 && vhc == 0) ? 2 : 0) - ev));
      if (vvalid) {
        uint32_t y[4], T[3];
#pragma unroll
        for (int j = 0; j < 4; ++j) y[j] = __float2uint_rn(W[j] * mult);
        transpose3(y, T);
#pragma unroll
        for (int dg = 0; dg < 6; ++dg) {
          const int ln = 4 * dg + vt;
          vb32[(ln * NG + swz(ln, vgp, NG)) * 2 + vhc] = digit4(T, dg);
        }
      }
      __syncwarp();
      uint2 vb[NG];
#pragma unroll
      for (int q = 0; q < NG; ++q) vb[q] = vbv[lane * NG + swz(lane, q, NG)];
      uint32_t vw[C::VWL];
#pragma unroll
      for (int q = 0; q < C::VWL / 4; ++q) {
        const uint4 x = reinterpret_cast<const uint4*>(vc)[q * 32 + lane];
        vw[4 * q] = x.x; vw[4 * q + 1] = x.y; vw[4 * q + 2] = x.z; vw[4 * q + 3] = x.w;
      }
#pragma unroll
      for (int mt = 0; mt < MTV; ++mt) {
        uint32_t a0, a1, a2, a3;
        if constexpr (BV == 2) {
          const uint32_t w = vw[mt], x = w >> 4;
          a0 = w & 0x03030303u; a2 = w & 0x0C0C0C0Cu;
          a1 = x & 0x03030303u; a3 = x & 0x0C0C0C0Cu;
        } else {
          const uint32_t w0 = vw[2 * mt], w1 = vw[2 * mt + 1];
          a0 = w0 & 0x0F0F0F0Fu; a1 = (w0 >> 4) & 0x0F0F0F0Fu;
          a2 = w1 & 0x0F0F0F0Fu; a3 = (w1 >> 4) & 0x0F0F0F0Fu;
        }
        mma_f8(acc[mt][0], a0, a1, a2, a3, vb[mt >> 1].x, vb[mt >> 1].y);
      }
      __syncwarp();
    } else {
      // ---- fp16 value path: items (token pair, group) -> raw p * s * F.
      // Fragment order (2/4-bit): item J = (gp, hk, tt, sp) covers tokens
      // 16 hk + 4 tt + sp + {0, 2}, the two halves of B register sp of lane tt
      // in k-step hk; F = 16 (codes as 1 + c/16) or 4 (2-bit codes at bits 2-3
      // of their byte, as 1 + c/4).  Sequential 8-bit: the Frag8 permutation.
      float raw[R][VJ][2];
      float zz[R][VJ];
      float vmax = 0.f;
#pragma unroll
      for (int i = 0; i < VJ; ++i) {
        const int J = lane + 32 * i;
        const int gp = J >> 4;
        int tau0, tau1;
        float f;
        if constexpr (C::VFRAG) {
          const int sp = J & 1, tt = (J >> 1) & 3, hk = (J >> 3) & 1;
          tau0 = 16 * hk + 4 * tt + sp;
          tau1 = tau0 + 2;
          f = (BV == 2 && hk) ? 4.f : 16.f;
        } else {
          const int P = J & 15;
          tau0 = 16 * (P >> 3) + Frag8::base(P & 7);
          tau1 = tau0 + Frag8::PARTNER;
          f = 1.f;
        }
        const bool valid = gp < NG;
        const float2 m0 = valid ? __half22float2(vm[tau0 * NG + gp]) : make_float2(0.f, 0.f);
        const float2 m1 = valid ? __half22float2(vm[tau1 * NG + gp]) : make_float2(0.f, 0.f);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float p0 = pb[r * 32 + tau0], p1 = pb[r * 32 + tau1];
          raw[r][i][0] = p0 * m0.x * f;
          raw[r][i][1] = p1 * m1.x * f;
          zz[r][i] = fmaf(p0, m0.y, p1 * m1.y);
          vmax = fmaxf(vmax, fmaxf(raw[r][i][0], raw[r][i][1]));
        }
      }
      // B_V = raw * 2^-ev must stay below 2^14; a trip (the first sub-block of a
      // pair, or larger weights/scales later) raises ev and rescales exactly.
      float fv = 1.f;
      if (__any_sync(0xffffffffu, vmax * pow2i(-ev) >= 16384.f)) {
        const float va = warp_max(vmax);
        const int evn = ilog2f(va) - 13;
        if (evn > ev) {
          fv = pow2i(max(ev - evn, -126));
          ev = evn;
        }
      }
      rescale(alpha, fv);
      {
        const float sv = pow2i(-ev), e2 = pow2i(ev);
#pragma unroll
        for (int i = 0; i < VJ; ++i) {
          const int J = lane + 32 * i;
          const int gp = J >> 4;
          int ks, slot_t, rg;
          if constexpr (C::VFRAG) {
            ks = (J >> 3) & 1;
            slot_t = (J >> 1) & 3;
            rg = J & 1;
          } else {
            const int P = J & 15, e0 = Frag8::base(P & 7);
            ks = P >> 3;
            slot_t = Frag8::lane_t(e0);
            rg = Frag8::reg(e0);
          }
          if (gp < NG) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
              const float v0 = raw[r][i][0] * sv, v1 = raw[r][i][1] * sv;
              const __half2 hi = __floats2half2_rn(v0, v1);
              const float2 hf = __half22float2(hi);
              const __half2 lo = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
              float cz = zz[r][i];
              if constexpr (C::VFRAG) {  // the constant 1 of 1 + c/F
                const float2 lf = __half22float2(lo);
                cz -= e2 * ((hf.x + lf.x) + (hf.y + lf.y));
              }
              corr[r][i] += cz;
              const int n0 = 2 * r, n1 = 2 * r + 1;
              vb32[(((gp * 2 + ks) * NT + (n0 >> 3)) * 32 + (n0 & 7) * 4 + slot_t) * 2 + rg] =
                  *reinterpret_cast<const uint32_t*>(&hi);
              vb32[(((gp * 2 + ks) * NT + (n1 >> 3)) * 32 + (n1 & 7) * 4 + slot_t) * 2 + rg] =
                  *reinterpret_cast<const uint32_t*>(&lo);
            }
          }
        }
      }
      __syncwarp();

      // O[c][2r+h] += sum_tok A_V[c][tok] * B_V[tok][2r+h]
      uint32_t vw[C::VFRAG ? C::VWL : 1];
      if constexpr (C::VFRAG) {
#pragma unroll
        for (int q = 0; q < C::VWL / 4; ++q) {
          const uint4 x = reinterpret_cast<const uint4*>(vc)[q * 32 + lane];
          vw[4 * q] = x.x; vw[4 * q + 1] = x.y; vw[4 * q + 2] = x.z; vw[4 * q + 3] = x.w;
        }
      }
#pragma unroll
      for (int mt = 0; mt < MTV; ++mt) {
        const int gp = mt >> 1;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          uint32_t a0, a1, a2, a3;
          if constexpr (C::VFRAG) {
            constexpr uint32_t ONE = 0x3C003C00u;
            if constexpr (BV == 2) {
              // row g: bits 8j (k-step 0) / 8j+2 (k-step 1); row g+8: +4.  Bytes
              // 0,2 give k-slots 2t, 2t+1; bytes 1,3 (w >> 8) give 2t+8, 2t+9.
              const uint32_t w = vw[mt], y = w >> 8;
              const uint32_t M = ks ? 0x03000300u : 0x00C000C0u;
              a0 = ((w << 6) & M) | ONE;
              a1 = ((w << 2) & M) | ONE;
              a2 = ((y << 6) & M) | ONE;
              a3 = ((y << 2) & M) | ONE;
            } else {
              const uint32_t w = vw[2 * mt + ks], y = w >> 8;
              constexpr uint32_t M = 0x03C003C0u;
              a0 = ((w << 6) & M) | ONE;
              a1 = ((w << 2) & M) | ONE;
              a2 = ((y << 6) & M) | ONE;
              a3 = ((y << 2) & M) | ONE;
            }
          } else {
            const uint32_t* c0 = vc + (16 * mt + g) * BV;
            const uint32_t* c1 = c0 + 8 * BV;
            Frag8::get(c0 + ks * 4, t, a0, a2);
            Frag8::get(c1 + ks * 4, t, a1, a3);
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint2 b = vbv[((gp * 2 + ks) * NT + nt) * 32 + lane];
            mma_16816(acc[mt][nt], a0, a1, a2, a3, b.x, b.y);
          }
        }
      }
      __syncwarp();
    }
  };

  auto process_tail_chunk = [&](const uint8_t* st, int k) {
    const __half* kt = reinterpret_cast<const __half*>(st);
    const __half* vt = kt + TCH * D;
    const int t0 = k * TCH;
    const int n = min(TCH, p.T_t - t0);
    if constexpr (ROPE) {
      // key of tail token t at absolute position T_q + t, rotated after
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
      for (int j = 0; j < TCH; ++j) {
        if (j < n) {
          const float2* cs =
              p.rope_tab + static_cast<size_t>(p.T_q + t0 + j) * H + lane;
          float v[R];
#pragma unroll
          for (int r = 0; r < R; ++r) v[r] = 0.f;
#pragma unroll
          for (int f = 0; f < FPL; ++f) {
            const float2 c = cs[32 * f];
            const float k0 = __half2float(kt[j * D + lane + 32 * f]);
            const float k1 = __half2float(kt[j * D + lane + 32 * f + H]);
            const float r0 = k0 * c.x - k1 * c.y;
            const float r1 = k1 * c.x + k0 * c.y;
#pragma unroll
            for (int r = 0; r < R; ++r) v[r] = fmaf(qa[r][f], r0, fmaf(qb[r][f], r1, v[r]));
          }
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const float sj = warp_sum(v[r]);
            if (lane == j) pb[r * 32 + j] = sj;
          }
        }
      }
    } else {
      float qc[R][CPL];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int c = 0; c < CPL; ++c) qc[r][c] = os[r * D + lane * CPL + c];
#pragma unroll
      for (int j = 0; j < TCH; ++j) {
        if (j < n) {
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
          for (int r = 0; r < R; ++r) {
            float v = 0.f;
#pragma unroll
            for (int c = 0; c < CPL; ++c) v = fmaf(qc[r][c], kk[c], v);
            const float sj = warp_sum(v);
            if (lane == j) pb[r * 32 + j] = sj;
          }
        }
      }
    }
    __syncwarp();
    float sc[R], mx[R], alpha[R], mnew[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      sc[r] = lane < n ? pb[r * 32 + lane] : -INFINITY;
      mx[r] = warp_max(sc[r]);
    }
    softmax_merge(mx, alpha, mnew);
    rescale(alpha, 1.f);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float pj = fast_exp2(sc[r] - mnew[r]);
      l[r] = l[r] * alpha[r] + warp_sum(pj);
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


  auto write_partial = [&](int prr) {
    const long long pr = prr;
    const long long slot = gw + pr;
    if constexpr (C::VF8) {
      // digit columns 2t, 2t+1 of this lane -> value sums of channels
      // 16 mt + g (+ 8); the quad holds the six digits
      const float f0 = pow2i(8 * t), f1 = pow2i(8 * t + 4);
      const float e2 = pow2i((BV == 2 ? 16 : 18) + ev);
#pragma unroll
      for (int mt = 0; mt < MTV; ++mt) {
        float v0 = fmaf(acc[mt][0][0], f0, acc[mt][0][1] * f1);
        float v1 = fmaf(acc[mt][0][2], f0, acc[mt][0][3] * f1);
        v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
        v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
        v0 += __shfl_xor_sync(0xffffffffu, v0, 2);
        v1 += __shfl_xor_sync(0xffffffffu, v1, 2);
        if (t == 0) {
          os[16 * mt + g] = v0 * e2;
          os[16 * mt + 8 + g] = v1 * e2;
        }
      }
      // zero-point sums: item group vgp = lane >> 3 (eight lanes per group)
      float cg = corr[0][0];
      cg += __shfl_xor_sync(0xffffffffu, cg, 1);
      cg += __shfl_xor_sync(0xffffffffu, cg, 2);
      cg += __shfl_xor_sync(0xffffffffu, cg, 4);
      float ct[NG];
#pragma unroll
      for (int q = 0; q < NG; ++q) ct[q] = __shfl_sync(0xffffffffu, cg, 8 * q);
      __syncwarp();
      if (lane == 0) p.part_ml[slot] = make_float2(m[0], l[0]);
      float* o = p.part_o + slot * D + lane * CPL;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const int ch = lane * CPL + c;
        float cz = 0.f;
#pragma unroll
        for (int q = 0; q < NG; ++q)
          if (q == (ch >> 5)) cz = ct[q];
        o[c] = os[ch] + cz + acct[0][c];
      }
    } else {
      const float e2 = pow2i(ev);
      float ct[R][NG];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int k = 0; k < NG; ++k) {
          float v = 0.f;
#pragma unroll
          for (int i = 0; i < VJ; ++i)
            if (((lane + 32 * i) >> 4) == k) v += corr[r][i];
          ct[r][k] = warp_sum(v);
        }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int r = 4 * nt + t;
        if (r < R) {
#pragma unroll
          for (int mt = 0; mt < MTV; ++mt) {
            os[r * D + 16 * mt + g] = e2 * (acc[mt][nt][0] + acc[mt][nt][1]);
            os[r * D + 16 * mt + g + 8] = e2 * (acc[mt][nt][2] + acc[mt][nt][3]);
          }
        }
      }
      __syncwarp();
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (lane == 0) p.part_ml[slot * R + r] = make_float2(m[r], l[r]);
        float* o = p.part_o + (slot * R + r) * D + lane * CPL;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          const int ch = lane * CPL + c;
          float cz = 0.f;
#pragma unroll
          for (int k = 0; k < NG; ++k)
            if (k == (ch >> 5)) cz = ct[r][k];
          o[c] = os[r * D + ch] + cz + acct[r][c];
        }
      }
    }
    __syncwarp();
    if (p.fused) {
      // Publish this partial, take a ticket; the pair's last warp merges
      // (it never waits for the others: the ticket tells it they are done).
      __threadfence();
      __syncwarp();
      const long long x0 = pr * p.upp;
      const long long w0 = owner_warp(x0, p.U, p.n_warps);
      const long long w1 = owner_warp(x0 + p.upp - 1, p.U, p.n_warps);
      int last = 0;
      if (lane == 0) last = atomicAdd(&p.tickets[pr], 1) == static_cast<int>(w1 - w0);
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        __threadfence();
        // Lane i weighs partials i and i + 32; the partial rows are loaded
        // eight at a time before they are summed (one L2 round trip each).
        const int nseg = static_cast<int>(w1 - w0 + 1);  // <= 64 when fused
#pragma unroll 1
        for (int r = 0; r < R; ++r) {
          float2 a = make_float2(-INFINITY, 0.f), b = a;
          if (lane < nseg) a = __ldcg(&p.part_ml[(w0 + lane + pr) * R + r]);
          if (lane + 32 < nseg) b = __ldcg(&p.part_ml[(w0 + lane + 32 + pr) * R + r]);
          const float ms = warp_max(fmaxf(a.x, b.x));
          const float fa = fast_exp2(a.x - ms), fb = fast_exp2(b.x - ms);
          const float L = warp_sum(fmaf(fa, a.y, fb * b.y));
          float o[CPL];
#pragma unroll
          for (int c = 0; c < CPL; ++c) o[c] = 0.f;
#pragma unroll 1
          for (int wb = 0; wb < nseg; wb += 8) {
            float v[8][CPL];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const long long w = w0 + min(wb + u, nseg - 1);
              const float* src = p.part_o + ((w + pr) * R + r) * D + lane * CPL;
              if constexpr (CPL == 4) {
                const float4 x = __ldcg(reinterpret_cast<const float4*>(src));
                v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
              } else {
#pragma unroll
                for (int c = 0; c < CPL; ++c) v[u][c] = __ldcg(src + c);
              }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int w = wb + u;
              const float f = __shfl_sync(0xffffffffu, w < 32 ? fa : fb, w & 31);
              if (w < nseg) {
#pragma unroll
                for (int c = 0; c < CPL; ++c) o[c] = fmaf(f, v[u][c], o[c]);
              }
            }
          }
          const float inv = 1.f / L;
          float* dst = p.out + (pr * R + r) * D + lane * CPL;
#pragma unroll
          for (int c = 0; c < CPL; ++c) dst[c] = o[c] * inv;
        }
        if (lane == 0) p.tickets[pr] = 0;
      }
    }
  };

  // ---- main loop: unit n = u - ua sits in stage n % NS, phase (n / NS) & 1
  int pr = ua / upp;
  int j = ua - pr * upp;
  int s = 0;
  uint32_t ph = 0u;
  for (int u = ua; u < ub; ++u) {
    if (pr != cur) {
      if (cur >= 0) write_partial(cur);
      enter_pair(pr);
      cur = pr;
    }
    if (!mbar_wait_bounded(&bars[s], ph)) {
      // Give up: record the error, wait (bounded) for this warp's copies in
      // flight so no bulk copy lands after the CTA exits, and return.
      if (lane == 0) atomicExch(p.err, kDevErrWait);
      for (int k = u; k < lu; ++k)
        mbar_wait_bounded(&bars[(k - ua) % NS], static_cast<uint32_t>(((k - ua) / NS) & 1));
      return;
    }
    const uint8_t* st = ws + s * STAGE;
    if (j < nsub)
      process_sub(st, j);
    else
      process_tail_chunk(st, j - nsub);
    if (lu < ub) {
      if (lane == 0) issue(s);
      advance_load();
    }
    if (++s == NS) {
      s = 0;
      ph ^= 1u;
    }
    if (++j == upp) {
      j = 0;
      ++pr;
    }
  }
  if (cur >= 0) write_partial(cur);
}

template <int D, int BK, int BV, int R, bool ROPE>
cudaError_t decode_mma_prepare(int* ctas_per_sm) {
  using C = MmaCfg<D, BK, BV, R, ROPE>;
  cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<D, BK, BV, R, ROPE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      ctas_per_sm, decode_mma_kernel<D, BK, BV, R, ROPE>, kDecodeWarps * 32, C::SMEM);
}

template <int D, int BK, int BV, int R, bool ROPE>
cudaError_t decode_mma_launch(const DecodeParams& p, cudaStream_t stream) {
  using C = MmaCfg<D, BK, BV, R, ROPE>;
  const int grid = (p.n_warps + kDecodeWarps - 1) / kDecodeWarps;
  decode_mma_kernel<D, BK, BV, R, ROPE><<<grid, kDecodeWarps * 32, C::SMEM, stream>>>(p);
  return cudaGetLastError();
}

// Every (bits_k, bits_v) pair of the geometry (G = 32, keys per channel,
// values per token).
template <int D, int R, bool ROPE>
DecodeOps decode_mma_ops_for(int bk, int bv) {
#define KVQ_CASE(BK_, BV_)                                                              \
  if (bk == BK_ && bv == BV_)                                                           \
    return DecodeOps{decode_mma_prepare<D, BK_, BV_, R, ROPE>,                          \
                     decode_mma_launch<D, BK_, BV_, R, ROPE>};
  KVQ_CASE(2, 2) KVQ_CASE(2, 4) KVQ_CASE(2, 8)
  KVQ_CASE(4, 2) KVQ_CASE(4, 4) KVQ_CASE(4, 8)
  KVQ_CASE(8, 2) KVQ_CASE(8, 4) KVQ_CASE(8, 8)
#undef KVQ_CASE
  return DecodeOps{nullptr, nullptr};
}

// Defined in the per-(D, R) translation units; {nullptr, nullptr} when no
// tensor-core instantiation exists for (bk, bv, rope).
DecodeOps decode_mma_ops(int D, int R, int bk, int bv, bool rope);

}  // namespace kvq
