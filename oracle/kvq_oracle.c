/*
 * kvq_oracle.c — plain, slow CPU oracle of the low-bit KV-cache path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this library.  It shares no code, header, table
 * or constant with the CUDA library: every definition below is written out
 * again from the method's description and from the documented byte layout.
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off -fPIC -shared (no FMA
 * contraction, IEEE fp32 arithmetic, round-to-nearest-even).
 *
 * Sources of each step ("Your KV cache doesn't have a bit problem, it has a
 * geometry problem" = GEOMETRY; "Why KV Cache Geometry Matters More Than Bit
 * Precision" = DIAL):
 *   quantizer ........ GEOMETRY "What Quantization Error Is Actually Made Of";
 *                      DIAL "Inside the Attention Equation"
 *   key grouping ..... GEOMETRY "Keys: The Outliers Live in Fixed Channels"
 *   value grouping ... GEOMETRY "Values: Where the Intuition Breaks"
 *   fp16 tail ........ GEOMETRY "The Systems Tax, and Why It Is Not a Detail"
 *   RoPE after dequant GEOMETRY "Rotary Embeddings Complicate the Keys"
 *   attention ........ GEOMETRY "Values: Where the Intuition Breaks" (softmax
 *                      weighted sum of value vectors), evaluated in fp64.
 *   FP8 (E4M3) ....... "Rotate, Then Round: The Geometry of KV-Cache
 *                      Compression", "Key takeaway"; the OCP E4M3 format.
 *   outlier isolation  "Why KV Cache Geometry Matters More Than Bit
 *                      Precision", "KV Cache Size, GPU Memory Efficiency, and
 *                      the Shift to Geometry-Aware Quantization" (KVQuant);
 *                      GEOMETRY "Rotary Embeddings Complicate the Keys".
 *
 * Every function works on ONE (batch, kv-head) pair; loops are plain and in
 * the order of the definition.  Parity pins for every function live in the
 * CPU test suite (hand-worked ties, brute-force nearest-level search, golden
 * packed words, closed-form attention and RoPE cases).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- fp16 <-> fp32 (C _Float16: IEEE binary16, round to nearest even) ---- */

float kvo_h2f(uint16_t h) {
  _Float16 v;
  memcpy(&v, &h, 2);
  return (float)v;
}

uint16_t kvo_f2h(float f) {
  _Float16 v = (_Float16)f;
  uint16_t h;
  memcpy(&h, &v, 2);
  return h;
}

void kvo_h2f_array(const uint16_t* h, float* f, long n) {
  for (long i = 0; i < n; ++i) f[i] = kvo_h2f(h[i]);
}

void kvo_f2h_array(const float* f, uint16_t* h, long n) {
  for (long i = 0; i < n; ++i) h[i] = kvo_f2h(f[i]);
}

/* ---- the quantizer on one group ----------------------------------------- */

/* Quantizes the n fp16 values x[0], x[stride], ..., x[(n-1)*stride] with
 * `bits` bits.  The zero point is the smallest value, the step is the range
 * divided by 2^bits - 1 (rounded to fp16 for storage), and each element goes
 * to the nearest step, ties to even.  A stored step of 0 (range 0, or a step
 * below fp16's smallest subnormal) gives code 0 everywhere. */
void kvo_quantize_group(const uint16_t* x, long stride, int n, int bits,
                        uint16_t* scale_out, uint16_t* zero_out,
                        uint8_t* codes) {
  float mn = kvo_h2f(x[0]);
  float mx = mn;
  for (int i = 1; i < n; ++i) {
    float v = kvo_h2f(x[(long)i * stride]);
    if (v < mn) mn = v;
    if (v > mx) mx = v;
  }
  int levels = (1 << bits) - 1;
  float step = (mx - mn) / (float)levels;
  uint16_t s_h = kvo_f2h(step);
  float s = kvo_h2f(s_h);
  *scale_out = s_h;
  *zero_out = kvo_f2h(mn + 0.0f);
  for (int i = 0; i < n; ++i) {
    float v = kvo_h2f(x[(long)i * stride]);
    int c = 0;
    if (s != 0.0f) {
      float r = rintf((v - mn) / s);
      if (!(r >= 0.0f)) r = 0.0f;
      if (r > (float)levels) r = (float)levels;
      c = (int)r;
    }
    codes[i] = (uint8_t)c;
  }
}

/* ---- FP8 (E4M3) ------------------------------------------------------------
 * The 8-bit floating-point format E4M3 of the OCP 8-bit floating point
 * specification: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits.
 * Exponent field 0 holds zero and the subnormals m * 2^-9; there are no
 * infinities and S.1111.111 is NaN, so the largest finite magnitude is
 * S.1111.110 = 1.75 * 2^8 = 448.  An FP8 cache ("Rotate, Then Round: The
 * Geometry of KV-Cache Compression", "Key takeaway" and "In practice") stores
 * each element as E4M3 after dividing it by its group's scale. */

/* Value of an E4M3 code (NaN for the two NaN codes). */
float kvo_e4m3_value(uint8_t c) {
  int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  double v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
  return (float)(sign ? -v : v);
}

/* Nearest E4M3 code of a finite fp32 value, ties to the even mantissa;
 * magnitudes at or above 448 give +-448 (saturation).  The sign is kept,
 * also for values that round to zero. */
uint8_t kvo_e4m3_encode(float y) {
  int neg = signbit(y) ? 1 : 0;
  double a = fabs((double)y);
  uint8_t code;
  if (a >= 448.0) {
    code = 0x7E;
  } else {
    /* spacing of the representable values around a: 2^(e-3) in the binade
     * [2^e, 2^(e+1)) for e >= -6, and 2^-9 below 2^-6 (subnormals) */
    int e = -6;
    if (a >= ldexp(1.0, -6)) {
      frexp(a, &e);
      e -= 1;
    }
    double q = ldexp(1.0, e - 3);
    double v = rint(a / q) * q; /* a / q is exact; rint rounds half to even */
    if (v == 0.0) {
      code = 0;
    } else if (v < ldexp(1.0, -6)) {
      code = (uint8_t)(v / ldexp(1.0, -9));
    } else {
      int e2;
      frexp(v, &e2);
      e2 -= 1;
      code = (uint8_t)(((e2 + 7) << 3) | (int)((v / ldexp(1.0, e2) - 1.0) * 8.0));
    }
  }
  return neg ? (uint8_t)(code | 0x80) : code;
}

void kvo_e4m3_value_array(const uint8_t* c, float* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = kvo_e4m3_value(c[i]);
}

void kvo_e4m3_encode_array(const float* y, uint8_t* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = kvo_e4m3_encode(y[i]);
}

/* One group of an FP8 cache: scale = fp16(max |x| / 448) (IEEE fp32 divide,
 * then round to fp16), zero point 0, code = E4M3(x / scale) with the IEEE
 * fp32 quotient.  A stored scale of 0 gives code 0 everywhere. */
void kvo_quantize_group_fp8(const uint16_t* x, long stride, int n,
                            uint16_t* scale_out, uint16_t* zero_out,
                            uint8_t* codes) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float v = fabsf(kvo_h2f(x[(long)i * stride]));
    if (v > amax) amax = v;
  }
  uint16_t s_h = kvo_f2h(amax / 448.0f);
  float s = kvo_h2f(s_h);
  *scale_out = s_h;
  *zero_out = 0;
  for (int i = 0; i < n; ++i) {
    float v = kvo_h2f(x[(long)i * stride]);
    codes[i] = (s != 0.0f) ? kvo_e4m3_encode(v / s) : 0;
  }
}

/* ---- one tensor (K or V) of one pair ------------------------------------- */

/* X: fp16 [T][D].  Quantizes tokens [0, Tq), Tq = floor(T/G)*G.
 * codes: [Tq][D].  scale/zero: axis 0 (channel) -> [Tq/G][D], entry (i, d) is
 * channel d over tokens [i*G, (i+1)*G); axis 1 (token) -> [Tq][D/G], entry
 * (t, g) is token t over channels [g*G, (g+1)*G).  Returns Tq. */
static void quantize_group_fmt(const uint16_t* x, long stride, int n, int bits,
                               int fp8, uint16_t* scale_out, uint16_t* zero_out,
                               uint8_t* codes) {
  if (fp8)
    kvo_quantize_group_fp8(x, stride, n, scale_out, zero_out, codes);
  else
    kvo_quantize_group(x, stride, n, bits, scale_out, zero_out, codes);
}

int kvo_quantize_tensor(int T, int D, int G, int bits, int fp8, int axis,
                        const uint16_t* X, uint8_t* codes, uint16_t* scale,
                        uint16_t* zero) {
  int Tq = (T / G) * G;
  uint8_t* tmp = (uint8_t*)malloc((size_t)G);
  if (axis == 0) {
    for (int i = 0; i < Tq / G; ++i) {
      for (int d = 0; d < D; ++d) {
        const uint16_t* first = X + (size_t)(i * G) * D + d;
        quantize_group_fmt(first, D, G, bits, fp8, &scale[(size_t)i * D + d],
                           &zero[(size_t)i * D + d], tmp);
        for (int j = 0; j < G; ++j) codes[(size_t)(i * G + j) * D + d] = tmp[j];
      }
    }
  } else {
    int ng = D / G;
    for (int t = 0; t < Tq; ++t) {
      for (int g = 0; g < ng; ++g) {
        const uint16_t* first = X + (size_t)t * D + (size_t)g * G;
        quantize_group_fmt(first, 1, G, bits, fp8, &scale[(size_t)t * ng + g],
                           &zero[(size_t)t * ng + g], tmp);
        for (int j = 0; j < G; ++j) codes[(size_t)t * D + (size_t)g * G + j] = tmp[j];
      }
    }
  }
  free(tmp);
  return Tq;
}

/* ---- dequantization ------------------------------------------------------ */

/* out[t][d] = fmaf(value, scale, zero) in fp32, with the scale/zero entry the
 * axis selects; value is the integer code, or its E4M3 value for an FP8
 * cache. */
void kvo_dequantize_tensor(int Tq, int D, int G, int axis, int fp8,
                           const uint8_t* codes, const uint16_t* scale,
                           const uint16_t* zero, float* out) {
  for (int t = 0; t < Tq; ++t) {
    for (int d = 0; d < D; ++d) {
      size_t m = (axis == 0) ? (size_t)(t / G) * D + d
                             : (size_t)t * (D / G) + (size_t)(d / G);
      float s = kvo_h2f(scale[m]);
      float z = kvo_h2f(zero[m]);
      uint8_t c = codes[(size_t)t * D + d];
      float v = fp8 ? kvo_e4m3_value(c) : (float)c;
      out[(size_t)t * D + d] = fmaf(v, s, z);
    }
  }
}

/* ---- dense-and-sparse outlier isolation -----------------------------------
 * KVQuant's third ingredient besides per-channel keys and pre-RoPE keys
 * ("Why KV Cache Geometry Matters More Than Bit Precision", section "KV
 * Cache Size, GPU Memory Efficiency, and the Shift to Geometry-Aware
 * Quantization"; "Your KV cache doesn't have a bit problem, it has a geometry
 * problem", section "Rotary Embeddings Complicate the Keys"): a small
 * fraction of extreme values is kept apart, so that it does not widen the
 * step of its group ("Inside the Attention Equation": one very large
 * activation makes every element of its group coarser).  The pages give no
 * selection rule and no storage format.  Reading: in every G-token block of
 * a side, the n elements of largest magnitude (ties: lower token, then lower
 * channel) are kept exactly, in fp16, with their positions; every group
 * takes its minimum and maximum over its remaining elements (scale 0 and
 * zero +0 when none remain); the kept positions get code 0 and dequantize to
 * their kept value. */

/* kvo_quantize_group over the elements i with skip[i * skip_stride] == 0;
 * skipped elements get code 0. */
void kvo_quantize_group_masked(const uint16_t* x, long stride, int n, int bits,
                               const uint8_t* skip, long skip_stride,
                               uint16_t* scale_out, uint16_t* zero_out,
                               uint8_t* codes) {
  int any = 0;
  float mn = 0.0f, mx = 0.0f;
  for (int i = 0; i < n; ++i) {
    if (skip[(long)i * skip_stride]) continue;
    float v = kvo_h2f(x[(long)i * stride]);
    if (!any || v < mn) mn = v;
    if (!any || v > mx) mx = v;
    any = 1;
  }
  if (!any) {
    *scale_out = 0;
    *zero_out = 0;
    for (int i = 0; i < n; ++i) codes[i] = 0;
    return;
  }
  int levels = (1 << bits) - 1;
  float step = (mx - mn) / (float)levels;
  uint16_t s_h = kvo_f2h(step);
  float s = kvo_h2f(s_h);
  *scale_out = s_h;
  *zero_out = kvo_f2h(mn + 0.0f);
  for (int i = 0; i < n; ++i) {
    int c = 0;
    if (!skip[(long)i * skip_stride] && s != 0.0f) {
      float r = rintf((kvo_h2f(x[(long)i * stride]) - mn) / s);
      if (!(r >= 0.0f)) r = 0.0f;
      if (r > (float)levels) r = (float)levels;
      c = (int)r;
    }
    codes[i] = (uint8_t)c;
  }
}

/* Ordering of the selection: larger magnitude first, then lower position. */
static const uint16_t* g_sel_x;
static int by_magnitude(const void* a, const void* b) {
  int32_t i = *(const int32_t*)a, j = *(const int32_t*)b;
  float xi = fabsf(kvo_h2f(g_sel_x[i])), xj = fabsf(kvo_h2f(g_sel_x[j]));
  if (xi != xj) return xi > xj ? -1 : 1;
  return i < j ? -1 : (i > j ? 1 : 0);
}
static int ascending(const void* a, const void* b) {
  int32_t i = *(const int32_t*)a, j = *(const int32_t*)b;
  return i < j ? -1 : (i > j ? 1 : 0);
}

/* Positions (j*D + d) of the n elements of largest |x| in the G x D fp16
 * tile X (row stride D), in ascending order.  n <= G * D. */
void kvo_select_outliers(const uint16_t* X, int G, int D, int n, int32_t* pos) {
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)G * D);
  for (int i = 0; i < G * D; ++i) idx[i] = i;
  g_sel_x = X;
  qsort(idx, (size_t)G * D, sizeof(int32_t), by_magnitude);
  for (int k = 0; k < n; ++k) pos[k] = idx[k];
  qsort(pos, (size_t)n, sizeof(int32_t), ascending);
  free(idx);
}

/* kvo_quantize_tensor with n_out outliers isolated in every G-token block
 * (integer codes only).  outliers: [Tq/G][n_out] entries, each a uint32 with
 * the kept fp16 value in bits 0-15 and the position j*D + d inside the
 * block in bits 16-31, ascending by position.  Returns Tq. */
int kvo_quantize_tensor_sparse(int T, int D, int G, int bits, int axis, int n_out,
                               const uint16_t* X, uint8_t* codes, uint16_t* scale,
                               uint16_t* zero, uint32_t* outliers) {
  int Tq = (T / G) * G;
  uint8_t* skip = (uint8_t*)malloc((size_t)G * D);
  int32_t* pos = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_out > 0 ? n_out : 1));
  uint8_t* tmp = (uint8_t*)malloc((size_t)G);
  int ng = D / G;
  for (int i = 0; i < Tq / G; ++i) {
    const uint16_t* tile = X + (size_t)i * G * D;
    memset(skip, 0, (size_t)G * D);
    kvo_select_outliers(tile, G, D, n_out, pos);
    for (int k = 0; k < n_out; ++k) {
      skip[pos[k]] = 1;
      outliers[(size_t)i * n_out + k] = (uint32_t)tile[pos[k]] | ((uint32_t)pos[k] << 16);
    }
    if (axis == 0) {
      for (int d = 0; d < D; ++d) {
        kvo_quantize_group_masked(tile + d, D, G, bits, skip + d, D, &scale[(size_t)i * D + d],
                                  &zero[(size_t)i * D + d], tmp);
        for (int j = 0; j < G; ++j) codes[(size_t)(i * G + j) * D + d] = tmp[j];
      }
    } else {
      for (int j = 0; j < G; ++j) {
        for (int g = 0; g < ng; ++g) {
          size_t t = (size_t)i * G + j;
          kvo_quantize_group_masked(tile + (size_t)j * D + (size_t)g * G, 1, G, bits,
                                    skip + (size_t)j * D + (size_t)g * G, 1,
                                    &scale[t * ng + g], &zero[t * ng + g], tmp);
          for (int e = 0; e < G; ++e) codes[t * D + (size_t)g * G + e] = tmp[e];
        }
      }
    }
  }
  free(tmp);
  free(pos);
  free(skip);
  return Tq;
}

/* Dequantized values of the kept elements: out[i*G + pos / D][pos % D] =
 * their fp16 value, for every block i and entry. */
void kvo_apply_outliers(int Tq, int D, int G, int n_out, const uint32_t* outliers, float* out) {
  for (int i = 0; i < Tq / G; ++i) {
    for (int k = 0; k < n_out; ++k) {
      uint32_t e = outliers[(size_t)i * n_out + k];
      uint32_t p = e >> 16;
      out[((size_t)i * G + p / D) * D + p % D] = kvo_h2f((uint16_t)(e & 0xffff));
    }
  }
}

/* ---- the packed byte layout ---------------------------------------------- */

static void put_bits(uint8_t* base, size_t word_index, int bit, int bits,
                     unsigned value) {
  /* word `word_index` (little-endian uint32) gets `value` at bit `bit` */
  uint8_t* w = base + word_index * 4;
  uint32_t cur = (uint32_t)w[0] | ((uint32_t)w[1] << 8) |
                 ((uint32_t)w[2] << 16) | ((uint32_t)w[3] << 24);
  uint32_t mask = ((1u << bits) - 1u) << bit;
  cur = (cur & ~mask) | ((value << bit) & mask);
  w[0] = (uint8_t)(cur & 0xff);
  w[1] = (uint8_t)((cur >> 8) & 0xff);
  w[2] = (uint8_t)((cur >> 16) & 0xff);
  w[3] = (uint8_t)((cur >> 24) & 0xff);
}

static unsigned get_bits(const uint8_t* base, size_t word_index, int bit,
                         int bits) {
  const uint8_t* w = base + word_index * 4;
  uint32_t cur = (uint32_t)w[0] | ((uint32_t)w[1] << 8) |
                 ((uint32_t)w[2] << 16) | ((uint32_t)w[3] << 24);
  return (cur >> bit) & ((1u << bits) - 1u);
}

static void put_meta(uint8_t* base, size_t entry, uint16_t s, uint16_t z) {
  uint8_t* e = base + entry * 4;
  e[0] = (uint8_t)(s & 0xff);
  e[1] = (uint8_t)(s >> 8);
  e[2] = (uint8_t)(z & 0xff);
  e[3] = (uint8_t)(z >> 8);
}

static void get_meta(const uint8_t* base, size_t entry, uint16_t* s,
                     uint16_t* z) {
  const uint8_t* e = base + entry * 4;
  *s = (uint16_t)(e[0] | (e[1] << 8));
  *z = (uint16_t)(e[2] | (e[3] << 8));
}

/* A block: [K codes | K meta (4 D) | K outliers (4 n) | V codes | V meta
 * (4 D) | V outliers (4 n)], n the outliers kept per block side (0: no
 * outlier sections). */
size_t kvo_block_bytes_n(int D, int G, int bk, int bv, int n) {
  return (size_t)G * D * (bk + bv) / 8 + 8 * (size_t)D + 8 * (size_t)n;
}

size_t kvo_block_bytes(int D, int G, int bk, int bv) { return kvo_block_bytes_n(D, G, bk, bv, 0); }

/* offsets[0..5] = K codes, K meta, K outliers, V codes, V meta, V outliers */
void kvo_block_offsets_n(int D, int G, int bk, int bv, int n, size_t* offsets) {
  offsets[0] = 0;
  offsets[1] = (size_t)G * D * bk / 8;
  offsets[2] = offsets[1] + 4 * (size_t)D;
  offsets[3] = offsets[2] + 4 * (size_t)n;
  offsets[4] = offsets[3] + (size_t)G * D * bv / 8;
  offsets[5] = offsets[4] + 4 * (size_t)D;
}

/* offsets[0..3] = K codes, K meta, V codes, V meta (no outlier sections) */
void kvo_block_offsets(int D, int G, int bk, int bv, size_t* offsets) {
  size_t o[6];
  kvo_block_offsets_n(D, G, bk, bv, 0, o);
  offsets[0] = o[0];
  offsets[1] = o[1];
  offsets[2] = o[3];
  offsets[3] = o[4];
}

/* Which order a side's codes are stored in: 1 = fragment order, used when
 * keys are grouped per channel, values per token, G = 32 and D is 64 or 128
 * (any bit width); 0 = sequential order otherwise. */
int kvo_code_order(int D, int G, int bits, int ak, int av) {
  return (ak == 0 && av == 1 && G == 32 && (D == 64 || D == 128) &&
          (bits == 2 || bits == 4 || bits == 8)) ? 1 : 0;
}

/* Fragment order of one 32-token code region, seen as a tile of rows x cols
 * codes (keys: rows = the 32 tokens, cols = the D channels; values: rows =
 * the D channels, cols = the 32 tokens).  With
 *   row = 16*mt + 8*hr + g            (g < 8, hr < 2)
 *   col = 16*ks + 8*kh + 2*t + e      (t < 4, e < 2, kh < 2)
 * the code belongs to lane l = 4*g + t, in that lane's word
 *   w = mt*(cols/32) + ks/2   at bit 16*e + F2[hr][2*(ks%2) + kh]   (2 bits)
 *   w = mt*(cols/16) + ks     at bit 16*e + 8*kh + 4*hr             (4 bits)
 *   w = 2*(mt*(cols/16) + ks) + kh   at bit 8*(2*hr + e)            (8 bits)
 * with F2[0] = {0, 10, 12, 14} and F2[1] = {2, 4, 6, 8}, and word w of lane
 * l is word ((w/4)*32 + l)*4 + w%4 of the region. */
static void frag_position(int row, int col, int cols, int bits, size_t* word,
                          int* bit) {
  static const int F2[2][4] = {{0, 10, 12, 14}, {2, 4, 6, 8}};
  int mt = row / 16, hr = (row % 16) / 8, g = row % 8;
  int ks = col / 16, kh = (col % 16) / 8, t = (col % 8) / 2, e = col % 2;
  int lane = 4 * g + t;
  int w;
  if (bits == 2) {
    w = mt * (cols / 32) + ks / 2;
    *bit = 16 * e + F2[hr][2 * (ks % 2) + kh];
  } else if (bits == 4) {
    w = mt * (cols / 16) + ks;
    *bit = 16 * e + 8 * kh + 4 * hr;
  } else {
    w = 2 * (mt * (cols / 16) + ks) + kh;
    *bit = 8 * (2 * hr + e);
  }
  *word = ((size_t)(w / 4) * 32 + (size_t)lane) * 4 + (size_t)(w % 4);
}

/* Word and bit of key code (token j of the block, channel d).  Sequential
 * order: token-major rows of D*bk/32 words, channel d in word d/(32/bk) at
 * bit (d % (32/bk))*bk. */
static void key_position(int D, int G, int bk, int ak, int av, int j, int d,
                         size_t* word, int* bit) {
  if (kvo_code_order(D, G, bk, ak, av)) {
    frag_position(j, d, D, bk, word, bit);
  } else {
    int per = 32 / bk;
    *word = (size_t)j * (D * bk / 32) + (size_t)(d / per);
    *bit = (d % per) * bk;
  }
}

/* Word and bit of value code (token j of the block, channel d).  Sequential
 * order: 32-token chunks, channel-major inside a chunk, bv words per channel,
 * token j in word (j%32)/(32/bv) at bit ((j%32) % (32/bv))*bv. */
static void value_position(int D, int G, int bv, int ak, int av, int j, int d,
                           size_t* word, int* bit) {
  if (kvo_code_order(D, G, bv, ak, av)) {
    frag_position(d, j, 32, bv, word, bit);
  } else {
    int per = 32 / bv, c = j / 32, jj = j % 32;
    *word = ((size_t)c * D + d) * bv + (size_t)(jj / per);
    *bit = (jj % per) * bv;
  }
}

static void put_u32(uint8_t* base, size_t entry, uint32_t v) {
  uint8_t* e = base + entry * 4;
  e[0] = (uint8_t)(v & 0xff);
  e[1] = (uint8_t)((v >> 8) & 0xff);
  e[2] = (uint8_t)((v >> 16) & 0xff);
  e[3] = (uint8_t)((v >> 24) & 0xff);
}

static uint32_t get_u32(const uint8_t* base, size_t entry) {
  const uint8_t* e = base + entry * 4;
  return (uint32_t)e[0] | ((uint32_t)e[1] << 8) | ((uint32_t)e[2] << 16) | ((uint32_t)e[3] << 24);
}

/* Writes the Tq/G blocks of one pair into `blocks` (Tq/G * block bytes);
 * kout / vout: [Tq/G][n] outlier entries of each side (unused when n = 0). */
void kvo_pack_pair_n(int Tq, int D, int G, int bk, int bv, int ak, int av, int n,
                     const uint8_t* kcodes, const uint16_t* kscale,
                     const uint16_t* kzero, const uint8_t* vcodes,
                     const uint16_t* vscale, const uint16_t* vzero,
                     const uint32_t* kout, const uint32_t* vout, uint8_t* blocks) {
  size_t bb = kvo_block_bytes_n(D, G, bk, bv, n);
  size_t off[6];
  kvo_block_offsets_n(D, G, bk, bv, n, off);
  memset(blocks, 0, (size_t)(Tq / G) * bb);
  for (int i = 0; i < Tq / G; ++i) {
    uint8_t* blk = blocks + (size_t)i * bb;
    /* K codes, in the order kvo_code_order selects */
    for (int j = 0; j < G; ++j) {
      for (int d = 0; d < D; ++d) {
        size_t word;
        int bit;
        key_position(D, G, bk, ak, av, j, d, &word, &bit);
        put_bits(blk + off[0], word, bit, bk, kcodes[(size_t)(i * G + j) * D + d]);
      }
    }
    /* V codes, in the order kvo_code_order selects */
    for (int j = 0; j < G; ++j) {
      for (int d = 0; d < D; ++d) {
        size_t word;
        int bit;
        value_position(D, G, bv, ak, av, j, d, &word, &bit);
        put_bits(blk + off[3], word, bit, bv, vcodes[(size_t)(i * G + j) * D + d]);
      }
    }
    /* metadata: D entries each */
    for (int e = 0; e < D; ++e) {
      size_t km = (ak == 0) ? (size_t)i * D + e
                            : (size_t)(i * G + e / (D / G)) * (D / G) + e % (D / G);
      size_t vm = (av == 0) ? (size_t)i * D + e
                            : (size_t)(i * G + e / (D / G)) * (D / G) + e % (D / G);
      put_meta(blk + off[1], e, kscale[km], kzero[km]);
      put_meta(blk + off[4], e, vscale[vm], vzero[vm]);
    }
    /* outliers: n entries each */
    for (int k = 0; k < n; ++k) {
      put_u32(blk + off[2], k, kout[(size_t)i * n + k]);
      put_u32(blk + off[5], k, vout[(size_t)i * n + k]);
    }
  }
}

void kvo_pack_pair(int Tq, int D, int G, int bk, int bv, int ak, int av,
                   const uint8_t* kcodes, const uint16_t* kscale,
                   const uint16_t* kzero, const uint8_t* vcodes,
                   const uint16_t* vscale, const uint16_t* vzero,
                   uint8_t* blocks) {
  kvo_pack_pair_n(Tq, D, G, bk, bv, ak, av, 0, kcodes, kscale, kzero, vcodes, vscale, vzero,
                  NULL, NULL, blocks);
}

/* Inverse of kvo_pack_pair_n. */
void kvo_unpack_pair_n(int Tq, int D, int G, int bk, int bv, int ak, int av, int n,
                       const uint8_t* blocks, uint8_t* kcodes, uint16_t* kscale,
                       uint16_t* kzero, uint8_t* vcodes, uint16_t* vscale,
                       uint16_t* vzero, uint32_t* kout, uint32_t* vout) {
  size_t bb = kvo_block_bytes_n(D, G, bk, bv, n);
  size_t off[6];
  kvo_block_offsets_n(D, G, bk, bv, n, off);
  for (int i = 0; i < Tq / G; ++i) {
    const uint8_t* blk = blocks + (size_t)i * bb;
    for (int j = 0; j < G; ++j) {
      for (int d = 0; d < D; ++d) {
        size_t word;
        int bit;
        key_position(D, G, bk, ak, av, j, d, &word, &bit);
        kcodes[(size_t)(i * G + j) * D + d] = (uint8_t)get_bits(blk + off[0], word, bit, bk);
        value_position(D, G, bv, ak, av, j, d, &word, &bit);
        vcodes[(size_t)(i * G + j) * D + d] = (uint8_t)get_bits(blk + off[3], word, bit, bv);
      }
    }
    for (int e = 0; e < D; ++e) {
      size_t km = (ak == 0) ? (size_t)i * D + e
                            : (size_t)(i * G + e / (D / G)) * (D / G) + e % (D / G);
      size_t vm = (av == 0) ? (size_t)i * D + e
                            : (size_t)(i * G + e / (D / G)) * (D / G) + e % (D / G);
      get_meta(blk + off[1], e, &kscale[km], &kzero[km]);
      get_meta(blk + off[4], e, &vscale[vm], &vzero[vm]);
    }
    for (int k = 0; k < n; ++k) {
      kout[(size_t)i * n + k] = get_u32(blk + off[2], k);
      vout[(size_t)i * n + k] = get_u32(blk + off[5], k);
    }
  }
}

void kvo_unpack_pair(int Tq, int D, int G, int bk, int bv, int ak, int av,
                     const uint8_t* blocks, uint8_t* kcodes, uint16_t* kscale,
                     uint16_t* kzero, uint8_t* vcodes, uint16_t* vscale,
                     uint16_t* vzero) {
  kvo_unpack_pair_n(Tq, D, G, bk, bv, ak, av, 0, blocks, kcodes, kscale, kzero, vcodes, vscale,
                    vzero, NULL, NULL);
}

/* ---- RoPE (fp64) --------------------------------------------------------- */

/* Rotate-half RoPE at absolute position pos: for i < D/2 the channel pair
 * (i, i + D/2) turns by the angle pos * base^(-2i/D). */
void kvo_rope(double* x, int D, long pos, double base) {
  int h = D / 2;
  for (int i = 0; i < h; ++i) {
    double theta = pow(base, -2.0 * (double)i / (double)D);
    double a = (double)pos * theta;
    double c = cos(a), s = sin(a);
    double x0 = x[i], x1 = x[i + h];
    x[i] = x0 * c - x1 * s;
    x[i + h] = x1 * c + x0 * s;
  }
}

/* ---- attention (fp64) ----------------------------------------------------- */

/* One pair, R query heads.  Keys/values: tokens [0, Tq) from khat/vhat (fp32
 * [Tq][D]), then tokens [Tq, Tq + Tt) from ktail/vtail (fp16 [Tt][D]).
 * q: fp16 [R][D].  With rope != 0 key t is rotated at position t.
 * score_t = scale * sum_d q_d k_{t,d}; p = softmax(score); out = sum p_t v_t.
 * out: fp64 [R][D].  scores (optional, may be NULL): fp64 [R][Tq + Tt].
 * An empty sequence gives out = 0. */
void kvo_attention_pair(int R, int D, int Tq, int Tt, const uint16_t* q,
                        const float* khat, const float* vhat,
                        const uint16_t* ktail, const uint16_t* vtail,
                        double scale, int rope, double base, double* out,
                        double* scores) {
  int T = Tq + Tt;
  double* s = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
  double* k = (double*)malloc(sizeof(double) * (size_t)D);
  for (int r = 0; r < R; ++r) {
    for (int d = 0; d < D; ++d) out[(size_t)r * D + d] = 0.0;
    if (T == 0) continue;
    for (int t = 0; t < T; ++t) {
      for (int d = 0; d < D; ++d)
        k[d] = (t < Tq) ? (double)khat[(size_t)t * D + d]
                        : (double)kvo_h2f(ktail[(size_t)(t - Tq) * D + d]);
      if (rope) kvo_rope(k, D, t, base);
      double acc = 0.0;
      for (int d = 0; d < D; ++d)
        acc += (double)kvo_h2f(q[(size_t)r * D + d]) * k[d];
      s[t] = scale * acc;
      if (scores) scores[(size_t)r * T + t] = s[t];
    }
    double m = s[0];
    for (int t = 1; t < T; ++t)
      if (s[t] > m) m = s[t];
    double l = 0.0;
    for (int t = 0; t < T; ++t) {
      s[t] = exp(s[t] - m);
      l += s[t];
    }
    for (int t = 0; t < T; ++t) {
      double p = s[t] / l;
      for (int d = 0; d < D; ++d) {
        double v = (t < Tq) ? (double)vhat[(size_t)t * D + d]
                            : (double)kvo_h2f(vtail[(size_t)(t - Tq) * D + d]);
        out[(size_t)r * D + d] += p * v;
      }
    }
  }
  free(k);
  free(s);
}
