// kvq_device.cuh — device-side helpers and launch parameter blocks of the
// CUDA library (sm_103a).  Internal to csrc/.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kvq {

// Number of iterations of a bounded mbarrier wait before a kernel gives up,
// records KVQ_DEVERR_WAIT in the cache's error word and returns.  Each
// try_wait may suspend the thread for a hardware-chosen interval, so this is
// far above any legitimate wait (a few microseconds) and well below a hang.
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr int kDevErrWait = 1;

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// One-dimensional bulk copy global -> shared (TMA engine), completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on phase `parity` of `bar`: at most `limit` try_wait rounds.
// Returns false when the limit ran out (the caller records the error and
// stops).  A limit of 0 gives up at once (the fault-injection hook of the
// host API uses it; the drain of copies in flight always uses kWaitLimit).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint32_t limit = kWaitLimit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  return false;
}

// ---------------------------------------------------------------- code -> float

// Exact float value of a small unsigned code (< 2^23) without the
// quarter-rate integer-to-float converter: OR the code into the mantissa of
// 2^23 and subtract 2^23 (both steps exact).
__device__ __forceinline__ float code_to_float(uint32_t c) {
  return __int_as_float(0x4B000000u | c) - 8388608.0f;
}

// ---------------------------------------------------------------- FP8 (E4M3)

// Dispatch tag for a side stored as E4M3 (an 8-bit side of an FP8 cache).
constexpr int kBitsE4M3 = -8;

// E4M3 code of a finite fp32 value: nearest, ties to even, saturating at
// +-448 (the conversion instruction's satfinite mode).
__device__ __forceinline__ uint32_t e4m3_encode(float y) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3));
}

// Exact fp32 value of an E4M3 code.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const __half_raw h =
      __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c & 0xffu), __NV_E4M3);
  return __half2float(__half(h));
}

// Bytes 0 and 1 of v (two E4M3 codes) -> an exact fp16 pair, byte 0 in the
// low half.
__device__ __forceinline__ uint32_t e4m3x2_to_half2(uint32_t v) {
  const __half2_raw h =
      __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v & 0xffffu), __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

// Value of a code: the integer itself, or its E4M3 value.
template <bool F8>
__device__ __forceinline__ float code_value(uint32_t c) {
  if constexpr (F8) return e4m3_value(c);
  else return code_to_float(c);
}

// ---------------------------------------------------------------- warp reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---------------------------------------------------------------- parameter blocks

// The tensor-core decode kernel covers keys grouped per channel, values per
// token and G = 32 (a 32-token sub-block is then a whole block).
__host__ __device__ inline bool mma_geometry(int G, int ak, int av) {
  return ak == 0 && av == 1 && G == 32;
}

// Code order of one side (include/kvq.h, "Code order of a side"): fragment
// order for every bit width in the tensor-core geometry with D = 64 or 128,
// sequential order otherwise.
__host__ __device__ inline bool fragment_order(int D, int G, int bits, int ak, int av) {
  return mma_geometry(G, ak, av) && (D == 64 || D == 128) &&
         (bits == 2 || bits == 4 || bits == 8);
}

// Fragment order: word (within the side's 32-token region) and bit of tile
// element (row, col) of a tile with `cols` columns (keys: row = token, col =
// channel, cols = D; values: row = channel, col = token, cols = 32).
__host__ __device__ inline void frag_position(int row, int col, int cols, int bits, int* word,
                                              int* bit) {
  const int mt = row >> 4, hr = (row >> 3) & 1, g = row & 7;
  const int ks = col >> 4, kh = (col >> 3) & 1, t = (col >> 1) & 3, e = col & 1;
  int w;
  if (bits == 2) {
    const int pi = 2 * (ks & 1) + kh;  // F2[0] = {0, 10, 12, 14}, F2[1] = {2, 4, 6, 8}
    w = mt * (cols >> 5) + (ks >> 1);
    *bit = 16 * e + (hr ? 2 + 2 * pi : (pi ? 8 + 2 * pi : 0));
  } else if (bits == 4) {
    w = mt * (cols >> 4) + ks;
    *bit = 16 * e + 8 * kh + 4 * hr;
  } else {
    w = 2 * (mt * (cols >> 4) + ks) + kh;
    *bit = 8 * (2 * hr + e);
  }
  *word = ((w >> 2) * 32 + 4 * g + t) * 4 + (w & 3);
}

// Geometry of the packed cache, shared by all kernels.
struct CacheGeom {
  uint8_t* blocks;     // [P][NB][block_bytes]
  uint64_t block_bytes;
  int NB;              // blocks per pair
  int off_km, off_vc, off_vm;
  int D, G, bk, bv, ak, av;
  int P;
  int frag_k, frag_v;  // code order of each side: 1 fragment, 0 sequential
  int fp8;             // 1: both sides hold E4M3 codes with absmax scales
  int TC;              // rows per pair of a tail buffer (residual + G)
  int NSK;             // rows per pair of the sink window (n_sink)
  int nout;            // outliers kept per block and side (0: none)
  int off_ko, off_vo;  // the K and V outlier sections of a block
};

// ---------------------------------------------------------------- batch rows

// Batch rows whose sequences differ in length (a ragged cache) number at most
// kMaxRows; a uniform cache describes every row by row 0.
constexpr int kMaxRows = 64;

// Quantize / append / flush of one batch row (every pair of the row).  The
// row's n new tokens first fill its sink window (tokens [0, nsink) -> sink
// rows [sink0, sink0 + nsink)); the others follow its T_t tail rows as one
// combined sequence, whose first nflush * G tokens become blocks
// first_block, ... and whose tokens [rem_begin, rem_end) are copied into tail
// buffer `dst` from row dst_row0 on.
struct QuantRow {
  int n;
  int sink0, nsink;
  int T_t;
  int src, dst;        // tail buffer (0 or 1) read / written
  int nflush;
  int first_block;
  int rem_begin, rem_end, dst_row0;
};

// Quantize / append / flush launch: grid (max nflush + 1, P).  CTA x of pair
// p quantizes block x of its row's flush (x < nflush) or copies the row's
// remainder and sink tokens (x == nflush).
struct QuantParams {
  CacheGeom g;
  const __half* knew;  // pair p's new token r at row p * new_stride + r
  const __half* vnew;
  int new_stride;      // rows per pair of knew / vnew
  __half* ktail[2];    // the two tail buffers, [P][TC][D] each
  __half* vtail[2];
  __half* ksink;       // sink windows [P][NSK][D]
  __half* vsink;
  int ragged;          // 0: rows[0] describes every row
  int hkv;             // pairs per row
  QuantRow rows[kMaxRows];
};

// Dequantize launch: grid (T_q / G, P).
struct DequantParams {
  CacheGeom g;
  int T_q;
  float* kout;  // [P][T_q][D]
  float* vout;
};

// Tail tokens per unit of the tensor-core decode kernel: the fp16 tail is
// streamed through the same copy pipeline as the packed sub-blocks, in chunks
// whose K and V rows (2 * tch * D fp16 values) fill exactly one stage of
// D * (4 bk + 4 bv + 8) bytes.
__host__ __device__ constexpr int mma_tail_chunk(int bk, int bv) { return bk + bv + 2; }

// Units of `rows` fp16 rows (tail or sink window) of one pair: ceil(rows /
// tch) chunks for the tensor-core kernel, one unit for the CUDA-core kernel
// (tch = 0).
__host__ __device__ inline int fp16_units(int rows, int tch) {
  if (rows <= 0) return 0;
  return tch > 0 ? (rows + tch - 1) / tch : 1;
}

// The decode work as a flat sequence of units: pair p = b * hkv + h of row b
// owns units [first_unit(p), first_unit(p) + units_of_row(b)): its 32-token
// quantized sub-blocks, then its fp16 tail units, then its fp16 sink units.
// Token positions (RoPE): sink row t at t, quantized token i at Ts + i, tail
// row t at Ts + Tq + t.
//
// Warps split the work by cost: a pair costs its units plus `vcost` virtual
// units placed after its last unit, which stand for the work of leaving a
// pair (its partial, the merge, the next pair's query).  Warp w takes the
// costs [start(w), start(w+1)), start(w) = floor(w * C / W), and processes the
// real units among them; a warp whose costs are all virtual has no work.
struct UnitMap {
  int ragged;              // 0: row 0's counts hold for every row
  int hkv;                 // pairs per row
  int rows;                // row records in use (1 when uniform)
  int vcost;               // virtual cost units after every pair
  int U;                   // units of all pairs
  int C;                   // cost of all pairs (U + P * vcost)
  int W;                   // warps the costs are split over
  int cq, cr;              // C / W and C % W
  int Ts[kMaxRows];        // sink tokens of each row
  int Tq[kMaxRows];        // quantized tokens
  int Tt[kMaxRows];        // tail tokens, including those a fused append adds
  int ntu[kMaxRows];       // fp16 tail units of a pair of the row
  int upp[kMaxRows];       // units of a pair of the row
  int uoff[kMaxRows + 1];  // ragged: first unit of each row
  int coff[kMaxRows + 1];  // ragged: first cost of each row
};

// Fills ntu and upp of row b from its token counts (tch: fp16 rows per unit,
// 0 for one unit per fp16 region).
__host__ __device__ inline void set_row_units(UnitMap& m, int b, int tch) {
  m.ntu[b] = fp16_units(m.Tt[b], tch);
  m.upp[b] = m.Tq[b] / 32 + m.ntu[b] + fp16_units(m.Ts[b], tch);
}

// Host side, after set_row_units of every row record: the row offsets and
// totals for P = hkv * (ragged ? rows : batch) pairs, and the split over at
// most W warps (W is lowered to the unit count when that is smaller).
// Returns the warp count used.
inline int finish_map(UnitMap& m, int n_pairs, int vcost, long long W) {
  m.vcost = vcost;
  long long U = 0, C = 0;
  if (m.ragged) {
    m.uoff[0] = 0;
    m.coff[0] = 0;
    for (int b = 0; b < m.rows; ++b) {
      m.uoff[b + 1] = m.uoff[b] + m.hkv * m.upp[b];
      m.coff[b + 1] = m.coff[b] + m.hkv * (m.upp[b] + vcost);
    }
    U = m.uoff[m.rows];
    C = m.coff[m.rows];
  } else {
    U = static_cast<long long>(n_pairs) * m.upp[0];
    C = static_cast<long long>(n_pairs) * (m.upp[0] + vcost);
  }
  if (W > U) W = U;
  if (W < 1) W = 1;
  m.U = static_cast<int>(U);
  m.C = static_cast<int>(C);
  m.W = static_cast<int>(W);
  m.cq = static_cast<int>(C / W);
  m.cr = static_cast<int>(C % W);
  return m.W;
}

// Units, costs and pairs fit in 31 bits (kvq_create checks the cost of a
// full cache), so the lookups below divide in 32 bits.
__host__ __device__ inline int row_of(const UnitMap& m, long long pr) {
  if (!m.ragged) return 0;
  return static_cast<int>(pr) / m.hkv;
}

__host__ __device__ inline int units_of_row(const UnitMap& m, int b) { return m.upp[b]; }

__host__ __device__ inline long long first_unit(const UnitMap& m, long long pr) {
  const int p = static_cast<int>(pr);
  if (!m.ragged) return static_cast<long long>(p) * m.upp[0];
  const int b = p / m.hkv;
  return m.uoff[b] + static_cast<long long>(p - b * m.hkv) * m.upp[b];
}

// The pair that owns unit u (u < the total).
__host__ __device__ inline long long pair_of_unit(const UnitMap& m, long long u) {
  const int ui = static_cast<int>(u);
  if (!m.ragged) return ui / m.upp[0];
  int b = 0;
  while (m.uoff[b + 1] <= ui) ++b;
  return b * m.hkv + (ui - m.uoff[b]) / m.upp[b];
}

// The cost of the first unit of pair pr.
__host__ __device__ inline int first_cost(const UnitMap& m, long long pr) {
  const int p = static_cast<int>(pr);
  if (!m.ragged) return p * (m.upp[0] + m.vcost);
  const int b = p / m.hkv;
  return m.coff[b] + (p - b * m.hkv) * (m.upp[b] + m.vcost);
}

// The first real unit at or after cost c (0 <= c <= C): the unit of cost c,
// the next pair's first unit when c is one of a pair's virtual costs, U at C.
__host__ __device__ inline int unit_at_cost(const UnitMap& m, int c) {
  int b = 0, c0 = 0, u0 = 0;
  if (m.ragged) {
    while (b + 1 < m.rows && m.coff[b + 1] <= c) ++b;
    c0 = m.coff[b];
    u0 = m.uoff[b];
  }
  const int upp = m.upp[b];
  const int k = (c - c0) / (upp + m.vcost);
  const int j = c - c0 - k * (upp + m.vcost);
  return u0 + k * upp + (j < upp ? j : upp);
}

// First cost of warp w: floor(w * C / W), in 32-bit arithmetic.
__host__ __device__ inline int warp_cost(const UnitMap& m, int w) {
  return w * m.cq + (w * m.cr) / m.W;
}

// The real units [*ua, *ub) of warp w.
__host__ __device__ inline void warp_units(const UnitMap& m, int w, int* ua, int* ub) {
  *ua = unit_at_cost(m, warp_cost(m, w));
  *ub = unit_at_cost(m, warp_cost(m, w + 1));
}

// The warp that processes the unit of cost c: the largest w with
// start(w) <= c  <=>  w * C < (c + 1) * W.
__host__ __device__ __forceinline__ int owner_warp(const UnitMap& m, int c) {
  return static_cast<int>(((static_cast<long long>(c) + 1) * m.W - 1) / m.C);
}

// The warps [*w0, *w1] whose ranges hold units of pair pr (each writes one
// partial of the pair, into slot w + pr).
__host__ __device__ inline void pair_warps(const UnitMap& m, long long pr, int* w0, int* w1) {
  const int c0 = first_cost(m, pr);
  *w0 = owner_warp(m, c0);
  *w1 = owner_warp(m, c0 + units_of_row(m, row_of(m, pr)) - 1);
}

// Split-K decode launch.  Warp w of the grid processes its units of the unit
// map (warp_units) and writes one partial (m, l, o) per pair it touches into
// slot (w + p).
struct DecodeParams {
  CacheGeom g;
  UnitMap map;
  __half* ktail[2];     // the two tail buffers [P][TC][D]
  __half* vtail[2];
  unsigned long long act;  // bit b (bit 0 for a uniform cache): row b's tail is buffer 1
  const __half* ksink;  // sink windows [P][NSK][D]
  const __half* vsink;
  // Append fused into the decode (tensor-core kernel, no flush): the last
  // n_new tail rows of every pair are the tokens of knew/vnew
  // ([P][n_new][D]); the kernel also stores them into the pair's tail.
  int n_new;
  const __half* knew;
  const __half* vnew;
  int lg_G;             // log2(G)
  int lg_sub;           // log2(G / 32): 32-token sub-blocks per block
  int n_warps;          // warps of the launch (map.W)
  int rope;             // rotate keys after dequantization
  const float2* rope_tab;  // [max_ctx][D/2] {cos, sin}
  int rope_rows;        // rows of rope_tab (max_ctx)
  const __half* q;      // [P][R][D]
  float qscale;         // softmax scale * log2(e)
  float* part_o;        // [W + P][R][D]
  float2* part_ml;      // [W + P][R] {m, l} (m in log2 units)
  int* err;
  uint32_t wait_limit;  // try_wait rounds of a main-loop wait (kWaitLimit normally)
  // Fused merge: the last warp to finish a pair merges its partials into
  // `out` (ticket counters, one per pair, start and end at zero).
  int fused;
  int* tickets;         // [P]
  float* out;           // [P][R][D]
};

// The counts of pair pr that a decode kernel uses.
struct PairLens {
  int nsub, ntu, upp;   // 32-token sub-blocks, tail units, all units
  int Ts, Tq, Tt;       // token counts (Tt includes a fused append's tokens)
  int t_old;            // tail rows already stored (Tt - n_new)
  long long u0;         // first unit
  int buf;              // active tail buffer of the pair's row
};

__device__ __forceinline__ PairLens pair_lens(const DecodeParams& p, long long pr) {
  const int b = row_of(p.map, pr);
  PairLens l;
  l.Ts = p.map.Ts[b];
  l.Tq = p.map.Tq[b];
  l.Tt = p.map.Tt[b];
  l.t_old = l.Tt - p.n_new;
  l.nsub = l.Tq >> 5;
  l.ntu = p.map.ntu[b];
  l.upp = p.map.upp[b];
  l.u0 = first_unit(p.map, pr);
  l.buf = static_cast<int>((p.act >> b) & 1ull);
  return l;
}

// Sub-blocks and units of pair pr (the counts a decode loop tests per unit).
__device__ __forceinline__ int pair_nsub(const DecodeParams& p, long long pr) {
  return p.map.Tq[row_of(p.map, pr)] >> 5;
}
__device__ __forceinline__ int pair_upp(const DecodeParams& p, long long pr) {
  return p.map.upp[row_of(p.map, pr)];
}

// Walks a warp's units [u0, u1) in order as (pair, unit-in-pair) without
// dividing in the loop; the pair's counts are reloaded when it enters a pair.
struct UnitCursor {
  long long u, end;
  long long pr;
  int j;
  PairLens l;
  __device__ __forceinline__ void init(const DecodeParams& p, long long u0, long long u1) {
    u = u0;
    end = u1;
    pr = 0;
    j = 0;
    if (u < end) {
      pr = pair_of_unit(p.map, u);
      l = pair_lens(p, pr);
      j = static_cast<int>(u - l.u0);
    }
  }
  __device__ __forceinline__ void next(const DecodeParams& p) {
    ++u;
    if (++j == l.upp) {
      j = 0;
      ++pr;
      if (u < end) l = pair_lens(p, pr);
    }
  }
};

struct MergeParams {
  const float* part_o;
  const float2* part_ml;
  float* out;  // [P][R][D]
  UnitMap map;  // the decode launch's units and split
  int R, D;
};

// Two-level merge of the split partials (few pairs, many partials each):
// block (pair, query, chunk) merges at most CS partial slots into a level-2
// partial; the last block of a (pair, query), found with a ticket, merges the
// level-2 partials into the output.
// Rows (partial slots of a chunk, or chunks of a pair) one merge2 block
// merges at most (its shared-memory row table).
constexpr int kMerge2MaxRows = 512;

struct Merge2Params {
  const float* part_o;
  const float2* part_ml;
  float* lvl_o;    // [P*R*C2][D]
  float2* lvl_ml;  // [P*R*C2]
  int* tickets;    // [P*R], zero between launches
  float* out;      // [P][R][D]
  UnitMap map;     // the decode launch's units and split
  int R, D;
  int C2;          // level-1 chunks per (pair, query)
  int CS;          // partial slots per chunk
};


}  // namespace kvq
