// kvq_decode_mma.cuh — tensor-core decode attention for the pages' geometry
// (keys grouped per channel, values grouped per token, keys stored after
// RoPE), the configuration "Your KV cache doesn't have a bit problem, it has a
// geometry problem" recommends ("What to Do with This").
//
// Same work decomposition, TMA pipeline, partials and tail handling as
// decode_split_kernel; the per-sub-block arithmetic runs on mma.sync
// m16n8k16 (fp16 inputs, fp32 accumulation):
//
//   scores  S[token][n] = sum_c A_K[token][c] * B_K[c][n]
//           A_K = packed key codes turned into exact fp16 values, B_K = the
//           query folded with the per-channel key scale;
//   values  O[c][n]     = sum_tok A_V[c][tok] * B_V[tok][n]
//           A_V = packed value codes (channel-major words), B_V = the softmax
//           weight folded with the per-token value scale;
//   columns n = 2*r + h: query head r of the GQA group, h = 0/1 the high/low
//   fp16 halves of an fp32 operand (hi + lo keeps ~22 bits, so the products
//   carry fp32-level accuracy into the fp32 accumulators).
//
// Code -> fp16 conversion (one funnel shift and one LOP3 per code pair):
//   2-bit: a rotated code word gives, with two masks, the fp16 values
//          1 + c/4 (code at mantissa bits 8-9) and 1 + c/16 (bits 6-7);
//   4-bit: 1 + c/16 (code at mantissa bits 6-9);
//   8-bit: a byte permute builds 1024 + c, and one half2 subtraction of 1024
//          leaves the exact code.
// The constant 1 of the 2/4-bit encodings is removed with exact per-channel
// (keys) and per-token (values) corrections computed from the same fp16
// operands.  The code order inside a 16-element mma slice is a fixed
// permutation (Frag<B>::lane_t/reg/half) applied identically to both
// operands, so the contraction is unchanged.
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

// Code -> fp16 operand registers of one 16-element slice.  `w` points at the
// slice's words (BITS/2 of them).  x0 covers fragment columns (2t, 2t+1), x2
// covers (2t+8, 2t+9).  Element e of the slice sits in lane t = lane_t(e),
// register reg(e) (0 = x0/b0, 1 = x2/b1), half half(e); F(e) is the factor
// the other operand carries, OFF whether the encoding adds a constant 1.
// base(i) + {0, PARTNER}, i < 8, are the two elements (half 0 and half 1) of
// one register, so the other operand is written one 32-bit word at a time.
template <int BITS>
struct Frag;

template <>
struct Frag<2> {
  static constexpr bool OFF = true;
  static constexpr int PARTNER = 8;  // element sharing lane and register, other half
  __device__ static __forceinline__ int base(int i) { return i; }
  __device__ static __forceinline__ void get(const uint32_t* w, int t, uint32_t rot, uint32_t& x0,
                                             uint32_t& x2) {
    const uint32_t x = __funnelshift_r(w[0], w[0], rot);
    x0 = (x & 0x03000300u) | 0x3C003C00u;  // elements 2t+1, 2t+9 as 1 + c/4
    x2 = (x & 0x00C000C0u) | 0x3C003C00u;  // elements 2t,   2t+8 as 1 + c/16
  }
  __device__ static __forceinline__ int lane_t(int e) { return (e & 7) >> 1; }
  __device__ static __forceinline__ int reg(int e) { return (e & 1) ? 0 : 1; }
  __device__ static __forceinline__ int half(int e) { return e >= 8 ? 1 : 0; }
  __device__ static __forceinline__ float F(int e) { return (e & 1) ? 4.0f : 16.0f; }
};

template <>
struct Frag<4> {
  static constexpr bool OFF = true;
  static constexpr int PARTNER = 4;
  __device__ static __forceinline__ int base(int i) { return (i & 3) | ((i & 4) << 1); }
  __device__ static __forceinline__ void get(const uint32_t* w, int t, uint32_t rot, uint32_t& x0,
                                             uint32_t& x2) {
    const uint32_t x = __funnelshift_r(w[0], w[0], rot);
    const uint32_t y = __funnelshift_r(w[1], w[1], rot);
    x0 = (x & 0x03C003C0u) | 0x3C003C00u;  // elements t, t+4 as 1 + c/16
    x2 = (y & 0x03C003C0u) | 0x3C003C00u;  // elements 8+t, 12+t
  }
  __device__ static __forceinline__ int lane_t(int e) { return e & 3; }
  __device__ static __forceinline__ int reg(int e) { return e >= 8 ? 1 : 0; }
  __device__ static __forceinline__ int half(int e) { return (e & 7) >= 4 ? 1 : 0; }
  __device__ static __forceinline__ float F(int) { return 16.0f; }
};

template <>
struct Frag<8> {
  static constexpr bool OFF = false;
  static constexpr int PARTNER = 1;
  __device__ static __forceinline__ int base(int i) { return 2 * i; }
  __device__ static __forceinline__ void get(const uint32_t* w, int t, uint32_t, uint32_t& x0,
                                             uint32_t& x2) {
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
  __device__ static __forceinline__ int half(int e) { return e & 1; }
  __device__ static __forceinline__ float F(int) { return 1.0f; }
};

template <int D, int BK, int BV, int R, bool ROPE = false>
struct MmaCfg {
  static constexpr int NT = (2 * R + 7) / 8;  // n-tiles of 8 columns
  static constexpr int KS = D / 16;           // key slices (k-steps of the score mma)
  static constexpr int MT = D / 16;           // value m-tiles (16 channels)
  static constexpr int CPL = D / 32;
  static constexpr int KW = D * BK / 32;
  static constexpr int KC_S = 4 * D * BK;
  static constexpr int KM_S = 4 * D;
  static constexpr int VC_S = 4 * D * BV;
  static constexpr int VM_S = 4 * D;
  static constexpr int STAGE = KC_S + KM_S + VC_S + VM_S;
  static constexpr int NS = ROPE ? 2 : (STAGE <= 4096 ? 3 : 2);
  static constexpr int OFF_BAR = NS * STAGE;
  static constexpr int OFF_KF = OFF_BAR + 64;                 // [KS][NT][32] uint2
  static constexpr int OFF_VF = OFF_KF + KS * NT * 32 * 8;    // [4][2][NT][32] uint2
  static constexpr int OFF_PB = OFF_VF + 4 * 2 * NT * 32 * 8; // [R][32] float
  static constexpr int OFF_OS = OFF_PB + R * 32 * 4;          // [R][D] float
  // RoPE: per-warp key coefficients [R][D/2][8] floats; per-CTA table of
  // cos/sin(j * theta_i), j < 32, stored [D/2][32] float2.
  static constexpr int OFF_CF = OFF_OS + R * D * 4;
  static constexpr int WARP_BYTES = round_up(OFF_CF + (ROPE ? R * (D / 2) * 32 : 0), 128);
  static constexpr int CS_BYTES = ROPE ? (D / 2) * 32 * 8 : 0;
  static constexpr int SMEM = kDecodeWarps * WARP_BYTES + CS_BYTES;
};

template <int D, int BK, int BV, int R, bool ROPE>
__global__ void __launch_bounds__(kDecodeWarps * 32, R == 1 ? (ROPE ? 3 : 4) : (R <= 4 ? 3 : 1))
    decode_mma_kernel(const DecodeParams p) {
  using C = MmaCfg<D, BK, BV, R, ROPE>;
  using FK = Frag<BK>;
  using FV = Frag<BV>;
  constexpr int NS = C::NS, NT = C::NT, KS = C::KS, MT = C::MT, CPL = C::CPL;

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
  __half* kf = reinterpret_cast<__half*>(ws + C::OFF_KF);
  __half* vf = reinterpret_cast<__half*>(ws + C::OFF_VF);
  float* pb = reinterpret_cast<float*>(ws + C::OFF_PB);
  float* os = reinterpret_cast<float*>(ws + C::OFF_OS);

  const int G = p.g.G;
  const int lgG = p.lg_G;
  const int ng = D >> lgG;
  const int sub_mask = (1 << p.lg_sub) - 1;
  const long long ua = gw * p.U / p.n_warps;
  const long long ub = (gw + 1) * p.U / p.n_warps;
  const uint32_t rot = static_cast<uint32_t>(4 * t - 6) & 31u;

  // Fragment buffers: columns >= 2R are never written and stay zero.
  {
    uint32_t* z = reinterpret_cast<uint32_t*>(ws + C::OFF_KF);
    for (int i = lane; i < (C::OFF_PB - C::OFF_KF) / 4; i += 32) z[i] = 0u;
  }
  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  // Load cursor: the next quantized unit to copy (tail units are skipped).
  UnitCursor lc;
  lc.init(ua, p.upp);
  auto skip_tail = [&]() {
    while (lc.u < ub && lc.j == p.nsub) lc.next(p.upp);
  };
  auto issue = [&](long long pr, int j, int s) {
    const int blk = j >> p.lg_sub;
    const int ch = j & sub_mask;
    const uint8_t* base =
        p.g.blocks + (static_cast<size_t>(pr) * p.g.NB + blk) * p.g.block_bytes;
    uint8_t* st = ws + s * C::STAGE;
    const uint32_t vm_bytes = 128u * ng;  // 32 tokens x D/G entries
    mbar_arrive_expect_tx(&bars[s], C::KC_S + C::KM_S + C::VC_S + vm_bytes);
    bulk_g2s(st, base + ch * C::KC_S, C::KC_S, &bars[s]);
    bulk_g2s(st + C::KC_S, base + p.g.off_km, C::KM_S, &bars[s]);
    bulk_g2s(st + C::KC_S + C::KM_S, base + p.g.off_vc + ch * C::VC_S, C::VC_S, &bars[s]);
    bulk_g2s(st + C::KC_S + C::KM_S + C::VC_S, base + p.g.off_vm + ch * vm_bytes, vm_bytes,
             &bars[s]);
  };

  skip_tail();
  int issued = 0;
  for (int s = 0; s < NS && lc.u < ub; ++s) {
    if (lane == 0) issue(lc.pr, lc.j, s);
    ++issued;
    lc.next(p.upp);
    skip_tail();
  }

  // ---- state of the current pair
  // Key channels of this lane: KP pairs (c0, c0 + FK::PARTNER) that share one
  // fragment register, so each hi/lo split is one packed conversion.
  constexpr int KP = D / 64;
  // Value-operand jobs of this lane: (token pair, channel group), 16 token
  // pairs x up to 4 groups spread over 32 lanes.
  constexpr int VJ = 2;
  float qreg[R][KP][2];  // q * scale * log2(e)
  float m[R], l[R];      // online softmax, identical in all lanes
  float acc[MT][NT][4];
  float corr[R][VJ];     // value corrections of this lane's jobs
  float acct[R][CPL];    // fp16-tail contributions, channels lane*CPL + c
  int ev = -126;         // value operand exponent: B_V = p * s * F * 2^-ev
  long long cur = -1;
  int qi = 0;

  auto kchan = [&](int i, int h) {
    const int P = lane + 32 * i;
    return 16 * (P >> 3) + FK::base(P & 7) + h * FK::PARTNER;
  };

  auto enter_pair = [&](long long pr) {
    const __half* qp = p.q + static_cast<size_t>(pr) * R * D;
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
      for (int i = 0; i < KP; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) qreg[r][i][h] = __half2float(qp[r * D + kchan(i, h)]) * p.qscale;
      m[r] = -INFINITY;
      l[r] = 0.f;
#pragma unroll
      for (int k = 0; k < VJ; ++k) corr[r][k] = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) acct[r][c] = 0.f;
    }
#pragma unroll
    for (int a = 0; a < MT; ++a)
#pragma unroll
      for (int b = 0; b < NT; ++b)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[a][b][k] = 0.f;
    ev = -126;
    if constexpr (ROPE) {
      // the scaled query, all channels, for the rotated-key path
      for (int i = lane; i < R * D; i += 32) os[i] = __half2float(qp[i]) * p.qscale;
      __syncwarp();
    }
  };

  // value of f for this lane's accumulator columns (query 4*nt + t)
  auto lane_factor = [&](const float (&f)[R], int nt) -> float {
    float v = 1.f;
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (r == 4 * nt + t) v = f[r];
    return v;
  };

  // Multiplies the mma accumulators and corrections by per-query factors.
  auto rescale = [&](const float (&f)[R], float fv) {
    bool any = fv != 1.f;
#pragma unroll
    for (int r = 0; r < R; ++r) any |= f[r] != 1.f;
    if (!any) return;  // warp-uniform
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float lf = lane_factor(f, nt) * fv;
#pragma unroll
      for (int a = 0; a < MT; ++a)
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

  uint32_t* kf32 = reinterpret_cast<uint32_t*>(kf);
  uint32_t* vf32 = reinterpret_cast<uint32_t*>(vf);

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
      uint32_t kr[C::KW];
      {
        const uint4* row = reinterpret_cast<const uint4*>(kc + lane * C::KW);
#pragma unroll
        for (int v = 0; v < C::KW / 4; ++v) {
          const uint4 w4 = row[v];
          kr[4 * v] = w4.x; kr[4 * v + 1] = w4.y; kr[4 * v + 2] = w4.z; kr[4 * v + 3] = w4.w;
        }
      }
      constexpr int KPER = 32 / BK;
      constexpr uint32_t KMASK = (1u << BK) - 1u;
      float sc[R];
#pragma unroll
      for (int r = 0; r < R; ++r) sc[r] = 0.f;
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const float c0 = code_to_float((kr[i / KPER] >> ((i % KPER) * BK)) & KMASK);
        const float c1 = code_to_float((kr[(i + H) / KPER] >> (((i + H) % KPER) * BK)) & KMASK);
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
    // ---- key operand: B_K[c][2r+h] = hi/lo of q_r[c] * s_c * F(c) * 2^-ek
    float qh[R][KP][2];
    float kz[R];
    float amax = 0.f;
#pragma unroll
    for (int r = 0; r < R; ++r) kz[r] = 0.f;
#pragma unroll
    for (int i = 0; i < KP; ++i) {
      const float2 s0 = __half22float2(km[kchan(i, 0)]);
      const float2 s1 = __half22float2(km[kchan(i, 1)]);
      const float f = FK::F(FK::base((lane + 32 * i) & 7));
#pragma unroll
      for (int r = 0; r < R; ++r) {
        qh[r][i][0] = qreg[r][i][0] * s0.x * f;
        qh[r][i][1] = qreg[r][i][1] * s1.x * f;
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
      const int kk = P >> 3, e0 = FK::base(P & 7);
      const int slot_t = FK::lane_t(e0), rg = FK::reg(e0);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float v0 = qh[r][i][0] * sk, v1 = qh[r][i][1] * sk;
        const __half2 hi = __floats2half2_rn(v0, v1);
        const float2 hf = __half22float2(hi);
        const __half2 lo = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
        if (FK::OFF) {
          const float2 lf = __half22float2(lo);
          kz[r] -= ek2 * ((hf.x + lf.x) + (hf.y + lf.y));
        }
        const int n0 = 2 * r, n1 = 2 * r + 1;
        kf32[((kk * NT + (n0 >> 3)) * 32 + (n0 & 7) * 4 + slot_t) * 2 + rg] =
            *reinterpret_cast<const uint32_t*>(&hi);
        kf32[((kk * NT + (n1 >> 3)) * 32 + (n1 & 7) * 4 + slot_t) * 2 + rg] =
            *reinterpret_cast<const uint32_t*>(&lo);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) kz[r] = warp_sum(kz[r]);
    __syncwarp();

    // ---- scores: tokens 16*mt + g (c0,c1) and 16*mt + g + 8 (c2,c3)
    uint2 bk[KS][NT];
#pragma unroll
    for (int kk = 0; kk < KS; ++kk)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        bk[kk][nt] = reinterpret_cast<const uint2*>(kf)[(kk * NT + nt) * 32 + lane];
    float sc[2][NT][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < NT; ++b)
#pragma unroll
        for (int k = 0; k < 4; ++k) sc[a][b][k] = 0.f;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const uint32_t* r0 = kc + (16 * mt + g) * C::KW;
      const uint32_t* r1 = r0 + 8 * C::KW;
      if constexpr (BK <= 4) {
        uint32_t w0[C::KW], w1[C::KW];
#pragma unroll
        for (int v = 0; v < C::KW / 4; ++v) {
          const uint4 x = reinterpret_cast<const uint4*>(r0)[v];
          const uint4 y = reinterpret_cast<const uint4*>(r1)[v];
          w0[4 * v] = x.x; w0[4 * v + 1] = x.y; w0[4 * v + 2] = x.z; w0[4 * v + 3] = x.w;
          w1[4 * v] = y.x; w1[4 * v + 1] = y.y; w1[4 * v + 2] = y.z; w1[4 * v + 3] = y.w;
        }
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          uint32_t a0, a1, a2, a3;
          FK::get(&w0[kk * (BK / 2)], t, rot, a0, a2);
          FK::get(&w1[kk * (BK / 2)], t, rot, a1, a3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_16816(sc[mt][nt], a0, a1, a2, a3, bk[kk][nt].x, bk[kk][nt].y);
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          uint32_t a0, a1, a2, a3;
          FK::get(r0 + kk * (BK / 2), t, rot, a0, a2);
          FK::get(r1 + kk * (BK / 2), t, rot, a1, a3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_16816(sc[mt][nt], a0, a1, a2, a3, bk[kk][nt].x, bk[kk][nt].y);
        }
      }
    }

    // ---- online softmax (log2 units); lane holds query 4*nt + t
    float s4[NT][4];
    float mx[R], mxl[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float z = lane_factor(kz, nt);
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        s4[nt][2 * mt] = fmaf(ek2, sc[mt][nt][0] + sc[mt][nt][1], z);
        s4[nt][2 * mt + 1] = fmaf(ek2, sc[mt][nt][2] + sc[mt][nt][3], z);
      }
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

    // ---- value operand: jobs (token pair, group) -> raw p * s * F
    float raw[R][VJ][2];
    float zz[R][VJ];
    float vmax = 0.f;
#pragma unroll
    for (int i = 0; i < VJ; ++i) {
      const int J = lane + 32 * i;
      const int P = J & 15, gp = J >> 4;
      const int tau0 = 16 * (P >> 3) + FV::base(P & 7), tau1 = tau0 + FV::PARTNER;
      const float f = FV::F(FV::base(P & 7));
      const bool valid = gp < ng;
      const float2 m0 = valid ? __half22float2(vm[tau0 * ng + gp]) : make_float2(0.f, 0.f);
      const float2 m1 = valid ? __half22float2(vm[tau1 * ng + gp]) : make_float2(0.f, 0.f);
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
        const int P = J & 15, gp = J >> 4;
        if (gp < ng) {
          const int ks = P >> 3, e0 = FV::base(P & 7);
          const int slot_t = FV::lane_t(e0), rg = FV::reg(e0);
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const float v0 = raw[r][i][0] * sv, v1 = raw[r][i][1] * sv;
            const __half2 hi = __floats2half2_rn(v0, v1);
            const float2 hf = __half22float2(hi);
            const __half2 lo = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
            float cz = zz[r][i];
            if (FV::OFF) {
              const float2 lf = __half22float2(lo);
              cz -= e2 * ((hf.x + lf.x) + (hf.y + lf.y));
            }
            corr[r][i] += cz;
            const int n0 = 2 * r, n1 = 2 * r + 1;
            vf32[(((gp * 2 + ks) * NT + (n0 >> 3)) * 32 + (n0 & 7) * 4 + slot_t) * 2 + rg] =
                *reinterpret_cast<const uint32_t*>(&hi);
            vf32[(((gp * 2 + ks) * NT + (n1 >> 3)) * 32 + (n1 & 7) * 4 + slot_t) * 2 + rg] =
                *reinterpret_cast<const uint32_t*>(&lo);
          }
        }
      }
    }
    __syncwarp();

    // ---- values: O[c][2r+h] += sum_tok A_V[c][tok] * B_V[tok][2r+h]
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int gp = (16 * mt) >> lgG;
      const uint32_t* c0 = vc + (16 * mt + g) * BV;
      const uint32_t* c1 = c0 + 8 * BV;
      uint32_t w0[BV], w1[BV];
      if constexpr (BV == 2) {
        const uint2 x = *reinterpret_cast<const uint2*>(c0);
        const uint2 y = *reinterpret_cast<const uint2*>(c1);
        w0[0] = x.x; w0[1] = x.y; w1[0] = y.x; w1[1] = y.y;
      } else if constexpr (BV == 4) {
        const uint4 x = *reinterpret_cast<const uint4*>(c0);
        const uint4 y = *reinterpret_cast<const uint4*>(c1);
        w0[0] = x.x; w0[1] = x.y; w0[2] = x.z; w0[3] = x.w;
        w1[0] = y.x; w1[1] = y.y; w1[2] = y.z; w1[3] = y.w;
      }
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        uint32_t a0, a1, a2, a3;
        if constexpr (BV <= 4) {
          FV::get(&w0[ks * (BV / 2)], t, rot, a0, a2);
          FV::get(&w1[ks * (BV / 2)], t, rot, a1, a3);
        } else {
          FV::get(c0 + ks * (BV / 2), t, rot, a0, a2);
          FV::get(c1 + ks * (BV / 2), t, rot, a1, a3);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint2 b = reinterpret_cast<const uint2*>(vf)[((gp * 2 + ks) * NT + nt) * 32 + lane];
          mma_16816(acc[mt][nt], a0, a1, a2, a3, b.x, b.y);
        }
      }
    }
    __syncwarp();
  };

  // fp16 tail unit: lane = token for the scores (each lane issues its whole
  // key row as 16-byte loads at once), lane = channels for the values (the
  // value rows of up to 8 tokens are loaded before they are used).  The
  // query, scaled, sits in `os` (free until the pair's partial is written).
  auto process_tail = [&](long long pr) {
    const __half* kt = p.ktail + static_cast<size_t>(pr) * G * D;
    const __half* vt = p.vtail + static_cast<size_t>(pr) * G * D;
    const int d0 = lane * CPL;
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int i = 0; i < KP; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) os[r * D + kchan(i, h)] = qreg[r][i][h];
    __syncwarp();
    for (int t0 = 0; t0 < p.T_t; t0 += 32) {
      const int tk = t0 + lane;
      float sc[R];
#pragma unroll
      for (int r = 0; r < R; ++r) sc[r] = -INFINITY;
      if (tk < p.T_t) {
        const uint4* row = reinterpret_cast<const uint4*>(kt + static_cast<size_t>(tk) * D);
#pragma unroll
        for (int r = 0; r < R; ++r) sc[r] = 0.f;
        if constexpr (ROPE) {
          // rotate the fp16 key at its absolute position, then dot with q
          const float2* cs = p.rope_tab + static_cast<size_t>(p.T_q + tk) * (D / 2);
#pragma unroll 2
          for (int v = 0; v < D / 16; ++v) {
            const uint4 a4 = row[v], b4 = row[v + D / 16];
            const __half2* a2 = reinterpret_cast<const __half2*>(&a4);
            const __half2* b2 = reinterpret_cast<const __half2*>(&b4);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 ka = __half22float2(a2[e]), kb = __half22float2(b2[e]);
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int i = 8 * v + 2 * e + u;
                const float k0 = u ? ka.y : ka.x, k1 = u ? kb.y : kb.x;
                const float2 t2 = cs[i];
                const float r0 = k0 * t2.x - k1 * t2.y;
                const float r1 = k1 * t2.x + k0 * t2.y;
#pragma unroll
                for (int r = 0; r < R; ++r)
                  sc[r] = fmaf(os[r * D + i], r0, fmaf(os[r * D + i + D / 2], r1, sc[r]));
              }
            }
          }
        } else {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint4 kr[D / 16];
#pragma unroll
          for (int v = 0; v < D / 16; ++v) kr[v] = row[half * (D / 16) + v];
#pragma unroll
          for (int v = 0; v < D / 16; ++v) {
            const __half2* h2 = reinterpret_cast<const __half2*>(&kr[v]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 kk2 = __half22float2(h2[e]);
              const int d = 8 * (half * (D / 16) + v) + 2 * e;
#pragma unroll
              for (int r = 0; r < R; ++r) {
                const float2 q2 = *reinterpret_cast<const float2*>(os + r * D + d);
                sc[r] = fmaf(q2.x, kk2.x, fmaf(q2.y, kk2.y, sc[r]));
              }
            }
          }
        }
        }
      }
      float mx[R], alpha[R], mnew[R];
#pragma unroll
      for (int r = 0; r < R; ++r) mx[r] = warp_max(sc[r]);
      softmax_merge(mx, alpha, mnew);
      rescale(alpha, 1.f);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float pj = fast_exp2(sc[r] - mnew[r]);
        l[r] = l[r] * alpha[r] + warp_sum(pj);
        pb[r * 32 + lane] = pj;
      }
      __syncwarp();
      const int nt = min(32, p.T_t - t0);
      for (int j0 = 0; j0 < nt; j0 += 8) {
        float vv[8][CPL];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int tj = min(j0 + jj, nt - 1);
          const __half* vr = vt + static_cast<size_t>(t0 + tj) * D + d0;
          if constexpr (CPL == 4) {
            const uint2 x = *reinterpret_cast<const uint2*>(vr);
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&x.x));
            const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&x.y));
            vv[jj][0] = a.x; vv[jj][1] = a.y; vv[jj][2] = b.x; vv[jj][3] = b.y;
          } else {
#pragma unroll
            for (int c = 0; c < CPL; ++c) vv[jj][c] = __half2float(vr[c]);
          }
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          if (j0 + jj < nt) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
              const float pj = pb[r * 32 + j0 + jj];
#pragma unroll
              for (int c = 0; c < CPL; ++c) acct[r][c] = fmaf(pj, vv[jj][c], acct[r][c]);
            }
          }
        }
      }
      __syncwarp();
    }
  };

  auto write_partial = [&](long long pr) {
    const long long slot = gw + pr;
    const float e2 = pow2i(ev);
    float ct[R][4];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
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
        for (int mt = 0; mt < MT; ++mt) {
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
        for (int k = 0; k < 4; ++k)
          if (k == (ch >> lgG)) cz = ct[r][k];
        o[c] = os[r * D + ch] + cz + acct[r][c];
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
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float ms = -INFINITY;
          for (long long w = w0; w <= w1; ++w) ms = fmaxf(ms, __ldcg(&p.part_ml[(w + pr) * R + r]).x);
          float L = 0.f, o[CPL];
#pragma unroll
          for (int c = 0; c < CPL; ++c) o[c] = 0.f;
          for (long long w = w0; w <= w1; ++w) {
            const float2 ml = __ldcg(&p.part_ml[(w + pr) * R + r]);
            const float f = fast_exp2(ml.x - ms);
            L = fmaf(f, ml.y, L);
            const float* src = p.part_o + ((w + pr) * R + r) * D + lane * CPL;
#pragma unroll
            for (int c = 0; c < CPL; ++c) o[c] = fmaf(f, __ldcg(src + c), o[c]);
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

  UnitCursor uc;
  uc.init(ua, p.upp);
  for (; uc.u < ub; uc.next(p.upp)) {
    const long long pr = uc.pr;
    const int j = uc.j;
    if (pr != cur) {
      if (cur >= 0) write_partial(cur);
      enter_pair(pr);
      cur = pr;
    }
    if (j == p.nsub) {
      process_tail(pr);
      continue;
    }
    const int s = qi % NS;
    if (!mbar_wait_bounded(&bars[s], static_cast<uint32_t>((qi / NS) & 1))) {
      // Give up: record the error, wait (bounded) for this warp's copies in
      // flight so no bulk copy lands after the CTA exits, and return.
      if (lane == 0) atomicExch(p.err, kDevErrWait);
      for (int k = qi; k < issued; ++k)
        mbar_wait_bounded(&bars[k % NS], static_cast<uint32_t>((k / NS) & 1));
      return;
    }
    process_sub(ws + s * C::STAGE, j);
    ++qi;
    if (lc.u < ub) {
      if (lane == 0) issue(lc.pr, lc.j, s);
      ++issued;
      lc.next(p.upp);
      skip_tail();
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

template <int D, int R, bool ROPE>
DecodeOps decode_mma_ops_for(int bk, int bv) {
#define KVQ_CASE(BK_, BV_)                                                              \
  if (bk == BK_ && bv == BV_)                                                           \
    return DecodeOps{decode_mma_prepare<D, BK_, BV_, R, ROPE>,                          \
                     decode_mma_launch<D, BK_, BV_, R, ROPE>};
  KVQ_CASE(2, 2) KVQ_CASE(4, 4) KVQ_CASE(8, 8) KVQ_CASE(8, 4)
#undef KVQ_CASE
  return DecodeOps{nullptr, nullptr};
}

// Defined in the per-(D, R) translation units; {nullptr, nullptr} when no
// tensor-core instantiation exists for (bk, bv, rope).
DecodeOps decode_mma_ops(int D, int R, int bk, int bv, bool rope);

}  // namespace kvq
