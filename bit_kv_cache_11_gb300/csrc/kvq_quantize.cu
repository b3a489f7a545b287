// kvq_quantize.cu — prefill quantization, decode-time append with the tail
// flush, and the dequantize test path.
//
// The quantizer ("Your KV cache doesn't have a bit problem, it has a geometry
// problem", section "What Quantization Error Is Actually Made Of"): per group
// zero point = minimum, step = (max - min) / (2^B - 1), round each element to
// the nearest step.  Keys are grouped per channel over G tokens and values
// per token over G channels (sections "Keys: The Outliers Live in Fixed
// Channels", "Values: Where the Intuition Breaks"); both axes are selectable.
// The fp16 tail and its flush in whole groups follow section "The Systems
// Tax, and Why It Is Not a Detail".
//
// One CTA quantizes one G-token block of one (batch, kv-head) pair:
//   1. 16-byte loads of the block's G fp16 K rows and V rows into shared
//      memory (the rows come from the old tail or the new tokens);
//   2. one thread per quantization group (D key groups and D value groups
//      per block, whatever the axis): min/max -> fp32 step -> fp16 {scale,
//      zero} metadata, then the group's codes as bytes in shared memory,
//      rounded exactly as (x - min) / step with an IEEE divide would round;
//   3. one thread per output word packs 32/B byte codes and stores the word
//      (coalesced) in the block layout of include/kvq.h.
// The extra CTA x == nflush copies the remainder tokens into the tail.
//
// FP8 cache ("Rotate, Then Round: The Geometry of KV-Cache Compression",
// "Key takeaway"): the same groups, scale = fp16(max|x| / 448), zero 0, each
// element stored as the E4M3 code of x / scale.
#include "kvq_device.cuh"

namespace kvq {

namespace {

constexpr int kQuantThreads = 256;

// Row pitches of the shared tiles (padding keeps 16-byte accesses of
// neighbouring rows in different banks).
__host__ __device__ constexpr int xpitch(int D) { return D + 8; }   // halves
__host__ __device__ constexpr int kpitch(int D) { return D + 16; }  // bytes
__host__ __device__ constexpr int vpitch(int G) { return G + 16; }  // bytes

// Quantizer statistics of one group, kept in registers by the thread that
// owns the group: minimum, stored fp16 step (as fp32) and its correctly
// rounded reciprocal (0 when the step is 0).
struct Stat {
  float mn, s, rcp;
};

// Statistics from the group's minimum and maximum (exact fp16 values).
// FP8 cache: scale = fp16(max|x| / 448), zero 0 (mn and rcp unused).
__device__ __forceinline__ Stat stat_of(float mn, float mx, int bits, bool f8, __half2* meta_out) {
  if (f8) {
    const float amax = fmaxf(fabsf(mn), fabsf(mx));
    const __half s_h = __float2half_rn(__fdiv_rn(amax, 448.0f));
    *meta_out = __halves2half2(s_h, __float2half_rn(0.0f));
    return Stat{0.0f, __half2float(s_h), 0.0f};
  }
  // (mx - mn) + 0: a range of -0 (min and max zeros of opposite sign) is +0.
  const float range = __fadd_rn(__fsub_rn(mx, mn), 0.0f);
  const float step = __fdiv_rn(range, static_cast<float>((1 << bits) - 1));
  const __half s_h = __float2half_rn(step);
  const __half z_h = __float2half_rn(__fadd_rn(mn, 0.0f));  // a -0 minimum is stored as +0
  *meta_out = __halves2half2(s_h, z_h);
  const float s = __half2float(s_h);
  return Stat{mn, s, s == 0.0f ? 0.0f : __frcp_rn(s)};
}

// min/max over n values p[0], p[stride], ... (fp16 read exactly as fp32).
__device__ __forceinline__ Stat group_stat(const __half* x, int stride, int n, int bits, bool f8,
                                           __half2* meta_out) {
  float mn = __half2float(x[0]);
  float mx = mn;
  for (int i = 1; i < n; ++i) {
    const float v = __half2float(x[i * stride]);
    mn = fminf(mn, v);
    mx = fmaxf(mx, v);
  }
  return stat_of(mn, mx, bits, f8, meta_out);
}

// FP8 cache: code = E4M3(x / s) with the IEEE quotient; 0 when s is 0.
__device__ __forceinline__ uint32_t code_fp8(float x, const Stat& st) {
  return st.s == 0.0f ? 0u : e4m3_encode(__fdiv_rn(x, st.s));
}

// code = clamp(rintf((x - mn) / s), 0, 2^bits - 1) with the IEEE quotient,
// computed as (x - mn) * (1/s): for codes below 2^9 that product is within
// 2^-13 of the IEEE quotient, so unless it lies within 2^-12 of a rounding
// tie both round to the same integer; near a tie the IEEE divide decides.
// The near-tie case, out of line: a call taken only near a tie, instead of
// an IEEE divide the compiler would predicate into every element.
__device__ __noinline__ float tie_code(float d, float s) { return rintf(__fdiv_rn(d, s)); }

__device__ __forceinline__ uint32_t code_of(float x, const Stat& st, float top) {
  const float d = __fsub_rn(x, st.mn);
  float r = rintf(__fmul_rn(d, st.rcp));
  const float t = __fsub_rn(__fmul_rn(d, st.rcp), r);
  if (fabsf(t) > 0.5f - 0.000244140625f) r = tie_code(d, st.s);
  r = fminf(r, top);  // d >= 0 and rcp >= 0, so r >= 0 (+0 when s == 0)
  return __float_as_uint(r + 8388608.0f) & 0xffu;  // exact: r is an integer in [0, 255]
}

// ldmatrix of four 8x8 fp16 matrices (lane i addresses row i % 8 of matrix
// i / 8; 16-byte aligned rows): lane L receives row L / 4, columns 2 (L % 4)
// and 2 (L % 4) + 1 of each matrix; .trans: rows 2 (L % 4), 2 (L % 4) + 1 of
// column L / 4.
__device__ __forceinline__ void ldsm_x4(uint32_t (&x)[4], const __half* row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3])
               : "r"(smem_addr(row)));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&x)[4], const __half* row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3])
               : "r"(smem_addr(row)));
}

// code_of for the four elements of a slot (xa and xb: rows r0 and r1 at
// the same two columns, so the same statistics): q + 1.5 * 2^23 rounds q to
// the nearest integer, ties to even (rintf), into the low mantissa bits;
// one near-tie test covers the four elements; the steps are read only on
// that rare path.  Codes of xa come back in ca, of xb in cb (bits 0, 16).
__device__ __forceinline__ void code_quad(float2 xa, float2 xb, float4 st, const float2* ss,
                                          float top, uint32_t& ca, uint32_t& cb) {
  constexpr float kM = 12582912.0f;
  constexpr float kTie = 0.5f - 0.000244140625f;
  const float2 mn = make_float2(st.x, st.y), rc = make_float2(st.z, st.w);
  const float2 km = make_float2(kM, kM), nkm = make_float2(-kM, -kM), neg = make_float2(-1.f, -1.f);
  const float2 da = __fadd2_rn(xa, mn), db = __fadd2_rn(xb, mn);  // x - min, exactly
  const float2 qa = __fmul2_rn(da, rc), qb = __fmul2_rn(db, rc);
  float2 ma = __fadd2_rn(qa, km), mb = __fadd2_rn(qb, km);         // kM + rint(q)
  const float2 ta = __ffma2_rn(__fadd2_rn(ma, nkm), neg, qa);     // q - rint(q), exact
  const float2 tb = __ffma2_rn(__fadd2_rn(mb, nkm), neg, qb);
  if (fmaxf(fmaxf(fabsf(ta.x), fabsf(ta.y)), fmaxf(fabsf(tb.x), fabsf(tb.y))) > kTie) {
    const float2 s = *ss;
    if (fabsf(ta.x) > kTie) ma.x = tie_code(da.x, s.x) + kM;
    if (fabsf(ta.y) > kTie) ma.y = tie_code(da.y, s.y) + kM;
    if (fabsf(tb.x) > kTie) mb.x = tie_code(db.x, s.x) + kM;
    if (fabsf(tb.y) > kTie) mb.y = tie_code(db.y, s.y) + kM;
  }
  const float hi = kM + top;  // r <= top exactly when kM + r <= kM + top
  // bytes {c0, 0, c1, 0}: kM + c has the code in byte 0 and a zero byte 1
  ca = __byte_perm(__float_as_uint(fminf(ma.x, hi)), __float_as_uint(fminf(ma.y, hi)), 0x1410);
  cb = __byte_perm(__float_as_uint(fminf(mb.x, hi)), __float_as_uint(fminf(mb.y, hi)), 0x1410);
}

// Row jc of pair p's combined sequence (its row's tail rows, then the new
// tokens that follow the sink window's share), K or V.
__device__ __forceinline__ const __half* combined_row(const QuantParams& q, const QuantRow& r,
                                                      int p, int jc, bool isv) {
  const int D = q.g.D;
  if (jc < r.T_t) {
    const __half* t = isv ? (r.src ? q.vtail[1] : q.vtail[0]) : (r.src ? q.ktail[1] : q.ktail[0]);
    return t + (static_cast<size_t>(p) * q.g.TC + jc) * D;
  }
  return (isv ? q.vnew : q.knew) +
         (static_cast<size_t>(p) * q.new_stride + r.nsink + (jc - r.T_t)) * D;
}

// Packs 32/BITS byte codes (LSB-first order) into one word.
template <int BITS>
__device__ __forceinline__ uint32_t pack_word(const uint8_t* b);

template <>
__device__ __forceinline__ uint32_t pack_word<2>(const uint8_t* b) {
  const uint4 v = *reinterpret_cast<const uint4*>(b);
  // four 2-bit bytes b0..b3 -> b0 + 4 b1 + 16 b2 + 64 b3 in the top byte of
  // v * (2^24 + 2^18 + 2^12 + 2^6) (the lower partial products stay below 2^24)
  const uint32_t M = 0x01041040u;
  const uint32_t p0 = v.x * M, p1 = v.y * M, p2 = v.z * M, p3 = v.w * M;
  return __byte_perm(__byte_perm(p0, p1, 0x0073), __byte_perm(p2, p3, 0x0073), 0x5410);
}

template <>
__device__ __forceinline__ uint32_t pack_word<4>(const uint8_t* b) {
  const uint2 v = *reinterpret_cast<const uint2*>(b);
  uint32_t x = (v.x | (v.x >> 4)) & 0x00ff00ffu;
  uint32_t y = (v.y | (v.y >> 4)) & 0x00ff00ffu;
  x = (x | (x >> 8)) & 0xffffu;
  y = (y | (y >> 8)) & 0xffffu;
  return x | (y << 16);
}

template <>
__device__ __forceinline__ uint32_t pack_word<8>(const uint8_t* b) {
  return *reinterpret_cast<const uint32_t*>(b);
}

}  // namespace

// Shared ints of the outlier selection: two histograms (256 + 128), four
// results and a block scan's kQuantThreads / 32 + 1 slots.
constexpr int kSelectScratch = 256 + 128 + 4 + kQuantThreads / 32 + 1;

// Exclusive prefix sum of v over the CTA's kQuantThreads threads (tot: the
// sum of all); scratch holds kQuantThreads / 32 + 1 ints.  Ends with a CTA
// barrier, so scratch may be reused right after.
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* tot) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[wid] = x;
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int w = 0; w < kQuantThreads / 32; ++w) {
      const int t = scratch[w];
      scratch[w] = acc;
      acc += t;
    }
    scratch[kQuantThreads / 32] = acc;
  }
  __syncthreads();
  const int r = scratch[wid] + x - v;
  *tot = scratch[kQuantThreads / 32];
  __syncthreads();
  return r;
}

// The bucket b (searching from the top) where the running count of hist[]
// reaches `need` (need >= 1, sum(hist) >= need), and the count of elements
// in the buckets above b; one warp, nb buckets (a multiple of 32).
__device__ __forceinline__ void top_bucket(const int* hist, int nb, int need, int* b_out,
                                           int* above_out) {
  const int lane = threadIdx.x & 31;
  const int per = nb / 32;
  // lane l owns buckets [nb - (l+1) per, nb - l per): lane 0 the highest
  int sum = 0;
  for (int i = 0; i < per; ++i) sum += hist[nb - 1 - lane * per - i];
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, incl >= need);
  const int l = __ffs(hit) - 1;  // first lane whose prefix reaches need
  const int before = __shfl_sync(0xffffffffu, incl - sum, l);
  if (lane == l) {
    int acc = before;
    for (int i = 0; i < per; ++i) {
      const int b = nb - 1 - lane * per - i;
      if (acc + hist[b] >= need) {
        *b_out = b;
        *above_out = acc;
        break;
      }
      acc += hist[b];
    }
  }
}

// Dense-and-sparse isolation of one side of a block (G x D fp16 tile X, row
// pitch XP): the n elements of largest magnitude (ties: lower position
// j*D + d) get skip[pos] = 1 and an entry (fp16 bits | pos << 16), written
// in ascending position order to `entries` (global).  Every thread owns
// G*D / kQuantThreads consecutive positions.  sh: kSelectScratch ints of
// shared scratch.  Starts and ends with the CTA in step.
__device__ void select_outliers(const __half* X, int XP, int G, int D, int n, uint8_t* skip,
                                uint32_t* entries, int* sh) {
  const int tid = threadIdx.x;
  const int per = G * D / kQuantThreads;
  const int pos0 = tid * per;
  int* hist1 = sh;          // key >> 7
  int* hist2 = sh + 256;    // key & 127 within the chosen high bucket
  int* misc = sh + 384;     // [0] high bucket, [1] above it, [2] low bucket, [3] above it,
                            // [4, 4 + kQuantThreads / 32] the scans' scratch
  for (int i = tid; i < 384; i += kQuantThreads) sh[i] = 0;
  __syncthreads();
  auto key_at = [&](int pos) -> int {
    const int j = pos / D, d = pos - j * D;
    return __half_as_ushort(X[j * XP + d]) & 0x7fff;
  };
  for (int i = 0; i < per; ++i) atomicAdd(&hist1[key_at(pos0 + i) >> 7], 1);
  __syncthreads();
  if (tid < 32) top_bucket(hist1, 256, n, &misc[0], &misc[1]);
  __syncthreads();
  const int b1 = misc[0];
  for (int i = 0; i < per; ++i) {
    const int k = key_at(pos0 + i);
    if ((k >> 7) == b1) atomicAdd(&hist2[k & 127], 1);
  }
  __syncthreads();
  if (tid < 32) top_bucket(hist2, 128, n - misc[1], &misc[2], &misc[3]);
  __syncthreads();
  const int T = (b1 << 7) | misc[2];       // the n-th largest key
  const int need = n - misc[1] - misc[3];  // how many elements equal to T are kept
  int eq = 0;
  for (int i = 0; i < per; ++i) eq += key_at(pos0 + i) == T;
  int tot;
  int rank = block_exclusive_scan(eq, misc + 4, &tot);
  int kept = 0;
  for (int i = 0; i < per; ++i) {
    const int k = key_at(pos0 + i);
    bool keep = k > T;
    if (k == T) keep = rank++ < need;
    skip[pos0 + i] = keep ? 1 : 0;
    kept += keep;
  }
  const int base = block_exclusive_scan(kept, misc + 4, &tot);
  int e = base;
  for (int i = 0; i < per; ++i) {
    const int pos = pos0 + i;
    if (skip[pos]) {
      const int j = pos / D, d = pos - j * D;
      entries[e++] = static_cast<uint32_t>(__half_as_ushort(X[j * XP + d])) |
                     (static_cast<uint32_t>(pos) << 16);
    }
  }
  __syncthreads();
}

// CTA x of pair p, whose row record is `row` (see QuantParams).
// Steps 2 and 3 for the pages' geometry (keys per channel, values per token,
// G = 32, fragment order on both sides, 2- or 4-bit codes, no outliers):
//   2. statistics only: thread c < D/2 takes key channels 2c, 2c+1 (fp16
//      min/max over the 32 rows), the next 32 * D/32 threads one value group
//      each; {min, 1/step} and the step go to shared memory, {scale, zero}
//      to the block;
//   3. one thread per output word, its lane the word's fragment lane: each
//      k-step's fp16 pairs come from one ldmatrix (.trans for the values),
//      the codes from code_quad, four at a time: no byte tile.
// The codes equal code_of's, element by element.
template <int BK, int BV, int D>
__device__ __forceinline__ void quantize_frag(const __half* xk, const __half* xv, float* sts,
                                              uint32_t* kc, __half2* kmeta, uint32_t* vc,
                                              __half2* vmeta) {
  constexpr int G = 32;
  constexpr int XP = xpitch(D);
  const int tid = threadIdx.x;
  constexpr int NG = D / G;
  float4* kst = reinterpret_cast<float4*>(sts);   // [D/2] {-mn, -mn', rcp, rcp'}
  float2* kss = reinterpret_cast<float2*>(kst + D / 2);          // [D/2] {s, s'}
  float4* vst = reinterpret_cast<float4*>(kss + D / 2);          // [NG][16]
  float2* vss = reinterpret_cast<float2*>(vst + NG * 16);        // [NG][16]
  if (tid < D / 2) {
    const __half2* col = reinterpret_cast<const __half2*>(xk) + tid;
    __half2 lo = col[0], hi = lo;
    for (int j = 1; j < G; ++j) {
      const __half2 h = col[j * (XP / 2)];
      lo = __hmin2(lo, h);
      hi = __hmax2(hi, h);
    }
    const Stat a = stat_of(__low2float(lo), __low2float(hi), BK, false, kmeta + 2 * tid);
    const Stat b = stat_of(__high2float(lo), __high2float(hi), BK, false, kmeta + 2 * tid + 1);
    kst[tid] = make_float4(-a.mn, -b.mn, a.rcp, b.rcp);
    kss[tid] = make_float2(a.s, b.s);
  } else if (tid < D / 2 + G * NG) {
    const int u = tid - D / 2, j = u & (G - 1), g = u >> 5;
    const __half* row = xv + j * XP + g * G;
    __half2 lo = *reinterpret_cast<const __half2*>(row), hi = lo;
#pragma unroll
    for (int i = 0; i < G; i += 8) {
      const uint4 v = *reinterpret_cast<const uint4*>(row + i);
      const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        lo = __hmin2(lo, h[k]);
        hi = __hmax2(hi, h[k]);
      }
    }
    const Stat st = stat_of(fminf(__low2float(lo), __high2float(lo)),
                            fmaxf(__low2float(hi), __high2float(hi)), BV, false, vmeta + j * NG + g);
    float* f = reinterpret_cast<float*>(vst + g * 16 + (j >> 1));
    f[j & 1] = -st.mn;
    f[2 + (j & 1)] = st.rcp;
    reinterpret_cast<float*>(vss + g * 16 + (j >> 1))[j & 1] = st.s;
  }
  __syncthreads();

  // K words (tile: 32 token rows x D channels), then V words (D channel
  // rows x 32 tokens).  Warp w takes lane words lw = w, w + 8, ...; its lane
  // is the word's fragment lane, so one ldmatrix (.trans for the values,
  // whose tile is stored token-major) hands every lane the fp16 pairs of a
  // k-step: registers 0 and 1 rows r0 and r1 at columns 2t, 2t + 1, 2 and 3
  // the same at columns 2t + 8, 2t + 9.  Bit widths are compile-time.
  constexpr float topk = static_cast<float>((1 << BK) - 1), topv = static_cast<float>((1 << BV) - 1);
  constexpr int lgk = (BK == 2 ? 0 : 1) + (D == 128 ? 2 : 1);  // log2(D * BK / 64)
  constexpr int lgv = BV == 2 ? 0 : 1;
  constexpr int NWARP = kQuantThreads / 32;
  const int lane = tid & 31, warp = tid >> 5;
  const int t = lane & 3;
  const int lr = lane & 7, lm = lane >> 3;  // the row and matrix this lane addresses
  for (int lw = warp; lw < D * BK / 32; lw += NWARP) {
    const int mt = lw >> lgk, kk = lw & ((1 << lgk) - 1);
    uint32_t word = 0;
#pragma unroll
    for (int h = 0; h < (BK == 2 ? 2 : 1); ++h) {
      const int ks = BK == 2 ? 2 * kk + h : kk;
      uint32_t x[4];
      ldsm_x4(x, xk + (16 * mt + lr + 8 * (lm & 1)) * XP + 16 * ks + 8 * (lm >> 1));
#pragma unroll
      for (int kh = 0; kh < 2; ++kh) {
        // slot sl: bit offsets of rows r0 and r1
        const int sl = BK == 2 ? 2 * h + kh : kh;
        const int b0 = BK == 2 ? (sl ? 8 + 2 * sl : 0) : 8 * sl;
        const int b1 = BK == 2 ? 2 + 2 * sl : 8 * sl + 4;
        const int col = 16 * ks + 8 * kh + 2 * t;
        uint32_t ca, cb;
        code_quad(__half22float2(*reinterpret_cast<const __half2*>(&x[2 * kh])),
                  __half22float2(*reinterpret_cast<const __half2*>(&x[2 * kh + 1])), kst[col >> 1],
                  kss + (col >> 1), topk, ca, cb);
        word |= (ca << b0) | (cb << b1);
      }
    }
    kc[((lw >> 2) << 7) | (lane << 2) | (lw & 3)] = word;
  }
  for (int lw = warp; lw < D * BV / 32; lw += NWARP) {
    const int mt = lw >> lgv, kk = lw & ((1 << lgv) - 1);
    const int gv = mt >> 1;  // rows r0 = 16 mt + g and r1 = r0 + 8 share a channel group
    uint32_t word = 0;
#pragma unroll
    for (int h = 0; h < (BV == 2 ? 2 : 1); ++h) {
      const int ks = BV == 2 ? 2 * kk + h : kk;
      uint32_t x[4];
      ldsm_x4_trans(x, xv + (16 * ks + lr + 8 * (lm >> 1)) * XP + 16 * mt + 8 * (lm & 1));
#pragma unroll
      for (int kh = 0; kh < 2; ++kh) {
        const int sl = BV == 2 ? 2 * h + kh : kh;
        const int b0 = BV == 2 ? (sl ? 8 + 2 * sl : 0) : 8 * sl;
        const int b1 = BV == 2 ? 2 + 2 * sl : 8 * sl + 4;
        const int col = 16 * ks + 8 * kh + 2 * t;  // token
        uint32_t ca, cb;
        code_quad(__half22float2(*reinterpret_cast<const __half2*>(&x[2 * kh])),
                  __half22float2(*reinterpret_cast<const __half2*>(&x[2 * kh + 1])),
                  vst[gv * 16 + (col >> 1)], vss + gv * 16 + (col >> 1), topv, ca, cb);
        word |= (ca << b0) | (cb << b1);
      }
    }
    vc[((lw >> 2) << 7) | (lane << 2) | (lw & 3)] = word;
  }
}

// combined_row with the head dimension known at compile time.
template <int D>
__device__ __forceinline__ const __half* combined_row_d(const QuantParams& q, const QuantRow& r,
                                                        int p, int jc, bool isv) {
  if (jc < r.T_t) {
    const __half* t = isv ? (r.src ? q.vtail[1] : q.vtail[0]) : (r.src ? q.ktail[1] : q.ktail[0]);
    return t + (static_cast<size_t>(p) * q.g.TC + jc) * D;
  }
  return (isv ? q.vnew : q.knew) +
         (static_cast<size_t>(p) * q.new_stride + r.nsink + (jc - r.T_t)) * D;
}

// Block x (< row.nflush) of pair p in the pages' geometry (fragment order on
// both sides, G = 32, 2- or 4-bit codes, no outliers), the head dimension a
// compile-time constant: step 1 (the rows into shared memory) as in
// quantize_block, then quantize_frag.
template <int BK, int BV, int D>
__device__ __forceinline__ void quantize_block_frag(const QuantParams& q, const QuantRow& row, int x,
                                                    int p) {
  constexpr int G = 32, XP = xpitch(D), CPR = D / 8;  // 16-byte chunks per row
  const int tid = threadIdx.x;
  extern __shared__ __align__(16) uint8_t smem[];
  __half* xk = reinterpret_cast<__half*>(smem);
  __half* xv = xk + G * XP;
  float* sts = reinterpret_cast<float*>(xv + G * XP);
  constexpr int chunks = G * CPR;
  for (int c0 = tid; c0 < chunks; c0 += 2 * kQuantThreads) {
    uint4 rk[2], rv[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int c = c0 + k * kQuantThreads;
      if (c < chunks) {
        const int j = c / CPR, col = (c % CPR) * 8;
        rk[k] = *reinterpret_cast<const uint4*>(combined_row_d<D>(q, row, p, x * G + j, false) + col);
        rv[k] = *reinterpret_cast<const uint4*>(combined_row_d<D>(q, row, p, x * G + j, true) + col);
      }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int c = c0 + k * kQuantThreads;
      if (c < chunks) {
        const int j = c / CPR, col = (c % CPR) * 8;
        *reinterpret_cast<uint4*>(xk + j * XP + col) = rk[k];
        *reinterpret_cast<uint4*>(xv + j * XP + col) = rv[k];
      }
    }
  }
  __syncthreads();
  uint8_t* blk = q.g.blocks +
                 (static_cast<size_t>(p) * q.g.NB + row.first_block + x) * q.g.block_bytes;
  quantize_frag<BK, BV, D>(xk, xv, sts, reinterpret_cast<uint32_t*>(blk),
                           reinterpret_cast<__half2*>(blk + q.g.off_km),
                           reinterpret_cast<uint32_t*>(blk + q.g.off_vc),
                           reinterpret_cast<__half2*>(blk + q.g.off_vm));
}

// The extra CTA (x == nflush) of pair p: the remainder tokens into the tail,
// the first nsink new tokens into the sink window.
__device__ __forceinline__ void copy_remainder(const QuantParams& q, const QuantRow& row, int p) {
  const int D = q.g.D;
  const int tid = threadIdx.x;
  // remainder -> tail rows [dst_row0, ...) of buffer dst
  const int rows = row.rem_end - row.rem_begin;
  const int chunks = rows * (D / 8);
  for (int c = tid; c < chunks; c += blockDim.x) {
    const int r = c / (D / 8);
    const int col = (c % (D / 8)) * 8;
    const int jc = row.rem_begin + r;
    const size_t dst = (static_cast<size_t>(p) * q.g.TC + row.dst_row0 + r) * D + col;
    *reinterpret_cast<uint4*>(q.ktail[row.dst] + dst) =
        *reinterpret_cast<const uint4*>(combined_row(q, row, p, jc, false) + col);
    *reinterpret_cast<uint4*>(q.vtail[row.dst] + dst) =
        *reinterpret_cast<const uint4*>(combined_row(q, row, p, jc, true) + col);
  }
  // the first nsink new tokens -> sink rows [sink0, sink0 + nsink)
  const int schunks = row.nsink * (D / 8);
  for (int c = tid; c < schunks; c += blockDim.x) {
    const int r = c / (D / 8);
    const int col = (c % (D / 8)) * 8;
    const size_t src = (static_cast<size_t>(p) * q.new_stride + r) * D + col;
    const size_t dst = (static_cast<size_t>(p) * q.g.NSK + row.sink0 + r) * D + col;
    *reinterpret_cast<uint4*>(q.ksink + dst) = *reinterpret_cast<const uint4*>(q.knew + src);
    *reinterpret_cast<uint4*>(q.vsink + dst) = *reinterpret_cast<const uint4*>(q.vnew + src);
  }
}

template <int BK, int BV>
__device__ __forceinline__ void quantize_block(const QuantParams& q, const QuantRow& row, int x,
                                               int p) {
  const int D = q.g.D, G = q.g.G;
  const int tid = threadIdx.x;
  if (x > row.nflush) return;

  if (x == row.nflush) {
    copy_remainder(q, row, p);
    return;
  }

  extern __shared__ __align__(16) uint8_t smem[];
  const int XP = xpitch(D), KP = kpitch(D), VP = vpitch(G);
  __half* xk = reinterpret_cast<__half*>(smem);
  __half* xv = xk + G * XP;
  uint8_t* kcode = reinterpret_cast<uint8_t*>(xv + G * XP);  // [G][KP] token-major
  uint8_t* vcode = kcode + G * KP;                            // [D][VP] channel-major
  // outlier isolation: skip masks [G*D] per side and selection scratch
  const int nout = q.g.nout;
  uint8_t* kskip = vcode + D * VP;
  uint8_t* vskip = kskip + G * D;
  int* osh = reinterpret_cast<int*>(vskip + G * D);

  // 1. the block's rows (combined index x*G + j), 16-byte loads; two chunks
  // per side and thread are loaded before any is stored, so their latencies
  // overlap (the stores could otherwise alias the next loads)
  const int chunks = G * (D / 8);
  for (int c0 = tid; c0 < chunks; c0 += 2 * blockDim.x) {
    uint4 rk[2], rv[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int c = c0 + k * blockDim.x;
      if (c < chunks) {
        const int j = c / (D / 8);
        const int col = (c % (D / 8)) * 8;
        const int jc = x * G + j;
        rk[k] = *reinterpret_cast<const uint4*>(combined_row(q, row, p, jc, false) + col);
        rv[k] = *reinterpret_cast<const uint4*>(combined_row(q, row, p, jc, true) + col);
      }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int c = c0 + k * blockDim.x;
      if (c < chunks) {
        const int j = c / (D / 8);
        const int col = (c % (D / 8)) * 8;
        *reinterpret_cast<uint4*>(xk + j * XP + col) = rk[k];
        *reinterpret_cast<uint4*>(xv + j * XP + col) = rv[k];
      }
    }
  }
  __syncthreads();

  uint8_t* blk = q.g.blocks +
                 (static_cast<size_t>(p) * q.g.NB + row.first_block + x) * q.g.block_bytes;
  __half2* kmeta = reinterpret_cast<__half2*>(blk + q.g.off_km);
  __half2* vmeta = reinterpret_cast<__half2*>(blk + q.g.off_vm);

  // 1b. dense-and-sparse isolation: the nout elements of largest magnitude
  //     of each side are kept apart (skip masks) and stored as entries
  if (nout > 0) {
    select_outliers(xk, XP, G, D, nout, kskip, reinterpret_cast<uint32_t*>(blk + q.g.off_ko), osh);
    select_outliers(xv, XP, G, D, nout, vskip, reinterpret_cast<uint32_t*>(blk + q.g.off_vo), osh);
  }

  // 2. one thread per group: statistics, then the group's codes as bytes.
  //    Every block has D key groups and D value groups whatever the axis.
  int lgG = 5;
  while ((1 << lgG) < G) ++lgG;
  const int ng = D >> lgG;
  const bool f8 = BK == 8 && BV == 8 && q.g.fp8;
  auto code = [&](float v, const Stat& st, float top) -> uint8_t {
    return static_cast<uint8_t>(f8 ? code_fp8(v, st) : code_of(v, st, top));
  };
  for (int e = tid; e < 2 * D; e += blockDim.x) {
    const bool isv = e >= D;
    const int ee = isv ? e - D : e;
    const int axis = isv ? q.g.av : q.g.ak;
    const int bits = isv ? BV : BK;
    const float top = static_cast<float>((1 << bits) - 1);
    const __half* X = isv ? xv : xk;
    const uint8_t* skip = isv ? vskip : kskip;
    if (axis == 0 && nout > 0) {  // channel ee, its kept outliers excluded
      float mn = 0.f, mx = 0.f;
      bool any = false;
      for (int j = 0; j < G; ++j) {
        if (skip[j * D + ee]) continue;
        const float v = __half2float(X[j * XP + ee]);
        mn = any ? fminf(mn, v) : v;
        mx = any ? fmaxf(mx, v) : v;
        any = true;
      }
      const Stat st = stat_of(mn, mx, bits, f8, (isv ? vmeta : kmeta) + ee);
      for (int j = 0; j < G; ++j) {
        const uint8_t c = skip[j * D + ee] ? 0 : code(__half2float(X[j * XP + ee]), st, top);
        if (isv) vcode[ee * VP + j] = c;
        else kcode[j * KP + ee] = c;
      }
    } else if (axis == 0) {  // channel ee over the G tokens
      const Stat st = group_stat(X + ee, XP, G, bits, f8, (isv ? vmeta : kmeta) + ee);
      for (int j = 0; j < G; ++j) {
        const uint8_t c = code(__half2float(X[j * XP + ee]), st, top);
        if (isv) vcode[ee * VP + j] = c;
        else kcode[j * KP + ee] = c;
      }
    } else if (nout > 0) {  // token j, channels [g*G, (g+1)*G), kept outliers excluded
      const int j = ee & (G - 1), g = ee >> lgG;
      const __half* row = X + j * XP + (g << lgG);
      const uint8_t* sk = skip + j * D + (g << lgG);
      float mn = 0.f, mx = 0.f;
      bool any = false;
      for (int i = 0; i < G; ++i) {
        if (sk[i]) continue;
        const float v = __half2float(row[i]);
        mn = any ? fminf(mn, v) : v;
        mx = any ? fmaxf(mx, v) : v;
        any = true;
      }
      const Stat st = stat_of(mn, mx, bits, f8, (isv ? vmeta : kmeta) + j * ng + g);
      for (int i = 0; i < G; ++i) {
        const int d = (g << lgG) + i;
        const uint8_t c = sk[i] ? 0 : code(__half2float(row[i]), st, top);
        if (isv) vcode[d * VP + j] = c;
        else kcode[j * KP + d] = c;
      }
    } else {          // token j, channels [g*G, (g+1)*G); consecutive threads: consecutive j
      // the group's G contiguous values, 16 bytes at a time (row pitch 16 mod
      // 128 bytes: eight consecutive j cover all banks)
      const int j = ee & (G - 1), g = ee >> lgG;
      const __half* row = X + j * XP + (g << lgG);
      __half2 lo = *reinterpret_cast<const __half2*>(row), hi = lo;
      for (int i = 0; i < G; i += 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + i);
        const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          lo = __hmin2(lo, h[k]);
          hi = __hmax2(hi, h[k]);
        }
      }
      const Stat st = stat_of(fminf(__low2float(lo), __high2float(lo)),
                              fmaxf(__low2float(hi), __high2float(hi)), bits, f8,
                              (isv ? vmeta : kmeta) + j * ng + g);
      for (int i = 0; i < G; i += 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + i);
        const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __half22float2(h[k]);
          const int d = (g << lgG) + i + 2 * k;
          const uint8_t c0 = code(f.x, st, top);
          const uint8_t c1 = code(f.y, st, top);
          if (isv) {
            vcode[d * VP + j] = c0;
            vcode[(d + 1) * VP + j] = c1;
          } else {
            kcode[j * KP + d] = c0;
            kcode[j * KP + d + 1] = c1;
          }
        }
      }
    }
  }
  __syncthreads();

  // 3. pack and store.  Sequential order: K token-major rows; V 32-token
  // chunks, channel-major.  Fragment order (G = 32): word w of lane l = 4g + t
  // collects, per (hr, kh) and k-step, the two codes of tile row
  // 16 mt + 8 hr + g at columns 16 ks + 8 kh + 2 t + {0, 1} -- two adjacent
  // bytes of the code tile, spread to bits b and b + 16 (2 and 4 bits), or
  // kept as bytes 0-1 (row g) and 2-3 (row g + 8) of the word (8 bits).
  auto frag_word = [&](const uint8_t* tile, int pitch, int cols, int bits, int w) -> uint32_t {
    const int l = (w >> 2) & 31, lw = ((w >> 7) << 2) | (w & 3);
    const int g = l >> 2, t = l & 3;
    uint32_t word = 0;
    if (bits == 2) {
      const int mt = lw / (cols >> 5), kp = lw - mt * (cols >> 5);
#pragma unroll
      for (int hr = 0; hr < 2; ++hr)
#pragma unroll
        for (int pi = 0; pi < 4; ++pi) {  // pi = 2 * (ks % 2) + kh
          const int col = 16 * (2 * kp + (pi >> 1)) + 8 * (pi & 1) + 2 * t;
          const uint32_t two = *reinterpret_cast<const uint16_t*>(tile + (16 * mt + 8 * hr + g) * pitch + col);
          const int b = hr ? 2 + 2 * pi : (pi ? 8 + 2 * pi : 0);
          word |= __byte_perm(two, 0u, 0x7170) << b;  // bytes 0, 1 -> bits 0 and 16
        }
    } else if (bits == 4) {
      const int mt = lw / (cols >> 4), ks = lw - mt * (cols >> 4);
#pragma unroll
      for (int hr = 0; hr < 2; ++hr)
#pragma unroll
        for (int kh = 0; kh < 2; ++kh) {
          const int col = 16 * ks + 8 * kh + 2 * t;
          const uint32_t two = *reinterpret_cast<const uint16_t*>(tile + (16 * mt + 8 * hr + g) * pitch + col);
          word |= __byte_perm(two, 0u, 0x7170) << (8 * kh + 4 * hr);
        }
    } else {  // 8 bits: rows g and g + 8 at columns 2t, 2t + 1 of one k-half
      const int kh = lw & 1, q2 = lw >> 1;
      const int mt = q2 / (cols >> 4), ks = q2 - mt * (cols >> 4);
      const int col = 16 * ks + 8 * kh + 2 * t;
      const uint32_t lo = *reinterpret_cast<const uint16_t*>(tile + (16 * mt + g) * pitch + col);
      const uint32_t hi = *reinterpret_cast<const uint16_t*>(tile + (16 * mt + 8 + g) * pitch + col);
      word = lo | (hi << 16);
    }
    return word;
  };
  {
    constexpr int per = 32 / BK;
    const int kw = D * BK / 32;
    uint32_t* kc = reinterpret_cast<uint32_t*>(blk);
    for (int w = tid; w < G * kw; w += blockDim.x) {
      if (q.g.frag_k) {
        kc[w] = frag_word(kcode, KP, D, BK, w);
      } else {
        const int j = w / kw;
        kc[w] = pack_word<BK>(kcode + j * KP + (w - j * kw) * per);
      }
    }
  }
  {
    constexpr int per = 32 / BV;
    uint32_t* vc = reinterpret_cast<uint32_t*>(blk + q.g.off_vc);
    const int words = (G / 32) * D * BV;
    for (int w = tid; w < words; w += blockDim.x) {
      if (q.g.frag_v) {
        vc[w] = frag_word(vcode, VP, 32, BV, w);
      } else {
        const int c = w / (D * BV);
        const int rem = w - c * (D * BV);
        const int d = rem / BV;
        const int j0 = c * 32 + (rem - d * BV) * per;
        vc[w] = pack_word<BV>(vcode + d * VP + j0);
      }
    }
  }
}

// A uniform cache (RAGGED = false) reads row 0's record at a fixed parameter
// offset; a ragged one indexes the rows by the pair's batch row.
template <int BK, int BV, bool RAGGED>
__global__ void __launch_bounds__(kQuantThreads) quantize_kernel(const __grid_constant__ QuantParams q) {
  const int x = blockIdx.x;
  const int p = blockIdx.y;
  quantize_block<BK, BV>(q, q.rows[RAGGED ? p / q.hkv : 0], x, p);
}

// The pages' geometry (fragment order on both sides, G = 32, 2- or 4-bit
// codes, no outliers), head dimension D: a kernel of its own, so that its
// registers are not those of the general path.
template <int BK, int BV, int D, bool RAGGED>
__global__ void __launch_bounds__(kQuantThreads) quantize_frag_kernel(const __grid_constant__ QuantParams q) {
  const int x = blockIdx.x;
  const int p = blockIdx.y;
  const QuantRow& row = q.rows[RAGGED ? p / q.hkv : 0];
  if (x > row.nflush) return;
  if (x == row.nflush) {
    copy_remainder(q, row, p);
    return;
  }
  quantize_block_frag<BK, BV, D>(q, row, x, p);
}

__global__ void __launch_bounds__(kQuantThreads) dequantize_kernel(const DequantParams q) {
  const int i = blockIdx.x;
  const int p = blockIdx.y;
  const int D = q.g.D, G = q.g.G;
  const int ng = D / G;
  const uint8_t* blk =
      q.g.blocks + (static_cast<size_t>(p) * q.g.NB + i) * q.g.block_bytes;
  const uint32_t* kc = reinterpret_cast<const uint32_t*>(blk);
  const __half2* km = reinterpret_cast<const __half2*>(blk + q.g.off_km);
  const uint32_t* vc = reinterpret_cast<const uint32_t*>(blk + q.g.off_vc);
  const __half2* vm = reinterpret_cast<const __half2*>(blk + q.g.off_vm);
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int j = e / D, d = e % D;
    const size_t o = (static_cast<size_t>(p) * q.T_q + static_cast<size_t>(i) * G + j) * D + d;
    {
      const int bits = q.g.bk, per = 32 / bits;
      int w = j * (D * bits / 32) + d / per, bit = (d % per) * bits;
      if (q.g.frag_k) frag_position(j, d, D, bits, &w, &bit);
      const uint32_t c = (kc[w] >> bit) & ((1u << bits) - 1u);
      const float2 sz = __half22float2(km[q.g.ak == 0 ? d : j * ng + d / G]);
      q.kout[o] = fmaf(q.g.fp8 ? e4m3_value(c) : static_cast<float>(c), sz.x, sz.y);
    }
    {
      const int bits = q.g.bv, per = 32 / bits;
      const int ch = j / 32, jj = j % 32;
      int w = (ch * D + d) * bits + jj / per, bit = (jj % per) * bits;
      if (q.g.frag_v) frag_position(d, j, 32, bits, &w, &bit);
      const uint32_t c = (vc[w] >> bit) & ((1u << bits) - 1u);
      const float2 sz = __half22float2(vm[q.g.av == 0 ? d : j * ng + d / G]);
      q.vout[o] = fmaf(q.g.fp8 ? e4m3_value(c) : static_cast<float>(c), sz.x, sz.y);
    }
  }
  // kept outliers replace their positions
  if (q.g.nout > 0) {
    __syncthreads();
    const uint32_t* ko = reinterpret_cast<const uint32_t*>(blk + q.g.off_ko);
    const uint32_t* vo = reinterpret_cast<const uint32_t*>(blk + q.g.off_vo);
    for (int k = threadIdx.x; k < 2 * q.g.nout; k += blockDim.x) {
      const bool isv = k >= q.g.nout;
      const uint32_t e = isv ? vo[k - q.g.nout] : ko[k];
      const int pos = static_cast<int>(e >> 16);
      const size_t o = (static_cast<size_t>(p) * q.T_q + static_cast<size_t>(i) * G + pos / D) * D +
                       pos % D;
      const float v = __half2float(__ushort_as_half(static_cast<unsigned short>(e & 0xffffu)));
      (isv ? q.vout : q.kout)[o] = v;
    }
  }
}

size_t quantize_smem_bytes(int D, int G, int nout) {
  size_t b = static_cast<size_t>(2) * G * xpitch(D) * sizeof(__half) +
             static_cast<size_t>(G) * kpitch(D) + static_cast<size_t>(D) * vpitch(G);
  if (nout > 0) b += static_cast<size_t>(2) * G * D + sizeof(int) * kSelectScratch;
  return b;
}

namespace {
using QuantFn = void (*)(const QuantParams);
QuantFn quant_fn(int bk, int bv, bool ragged) {
#define KVQ_Q(BK_, BV_) \
  if (bk == BK_ && bv == BV_)    \
    return ragged ? quantize_kernel<BK_, BV_, true> : quantize_kernel<BK_, BV_, false>;
  KVQ_Q(2, 2) KVQ_Q(2, 4) KVQ_Q(2, 8)
  KVQ_Q(4, 2) KVQ_Q(4, 4) KVQ_Q(4, 8)
  KVQ_Q(8, 2) KVQ_Q(8, 4) KVQ_Q(8, 8)
#undef KVQ_Q
  return nullptr;
}
QuantFn quant_frag_fn(int bk, int bv, int D, bool ragged) {
#define KVQ_QF(BK_, BV_, D_) \
  if (bk == BK_ && bv == BV_ && D == D_) \
    return ragged ? quantize_frag_kernel<BK_, BV_, D_, true> : quantize_frag_kernel<BK_, BV_, D_, false>;
  KVQ_QF(2, 2, 64) KVQ_QF(2, 4, 64) KVQ_QF(4, 2, 64) KVQ_QF(4, 4, 64)
  KVQ_QF(2, 2, 128) KVQ_QF(2, 4, 128) KVQ_QF(4, 2, 128) KVQ_QF(4, 4, 128)
#undef KVQ_QF
  return nullptr;
}
}  // namespace

// Opts every quantize instantiation into the shared memory of the largest
// block (G = D = 128); called once per cache creation, with its device current.
cudaError_t prepare_quantize() {
  const int bits[3] = {2, 4, 8};
  for (int a : bits)
    for (int b : bits)
      for (int rg = 0; rg < 2; ++rg) {
        cudaError_t e =
            cudaFuncSetAttribute(quant_fn(a, b, rg != 0), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(quantize_smem_bytes(128, 128, 0)));
        if (e != cudaSuccess) return e;
      }
  return cudaSuccess;
}

cudaError_t launch_quantize(const QuantParams& q, cudaStream_t stream) {
  const size_t smem = quantize_smem_bytes(q.g.D, q.g.G, q.g.nout);
  const bool frag = q.g.frag_k && q.g.frag_v && q.g.nout == 0 && q.g.bk != 8 && q.g.bv != 8;
  QuantFn fn = frag ? quant_frag_fn(q.g.bk, q.g.bv, q.g.D, q.ragged != 0)
                    : quant_fn(q.g.bk, q.g.bv, q.ragged != 0);
  if (fn == nullptr) return cudaErrorInvalidValue;
  int mx = 0;  // most blocks any row flushes
  const int nrows = q.ragged ? q.g.P / q.hkv : 1;
  for (int b = 0; b < nrows; ++b) mx = q.rows[b].nflush > mx ? q.rows[b].nflush : mx;
  dim3 grid(mx + 1, q.g.P);
  fn<<<grid, kQuantThreads, mx > 0 ? smem : 0, stream>>>(q);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const DequantParams& q, cudaStream_t stream) {
  dim3 grid(q.T_q / q.g.G, q.g.P);
  dequantize_kernel<<<grid, kQuantThreads, 0, stream>>>(q);
  return cudaGetLastError();
}

}  // namespace kvq
