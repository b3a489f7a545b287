/*
 * kvq.h — C ABI of the low-bit KV-cache library (one GPU, sm_103a).
 *
 * What it computes.  A key/value cache for one attention layer, stored with
 * uniform asymmetric integer quantization, and the decode attention that reads
 * that packed cache directly.
 *
 *   - The quantizer ("Your KV cache doesn't have a bit problem, it has a
 *     geometry problem", section "What Quantization Error Is Actually Made Of";
 *     also "Why KV Cache Geometry Matters More Than Bit Precision", section
 *     "Inside the Attention Equation"): per group, the zero point is the group
 *     minimum, the step is (max - min) / (2^B - 1), and every element is
 *     rounded to the nearest step.
 *   - The group geometry (same page, sections "Keys: The Outliers Live in Fixed
 *     Channels" and "Values: Where the Intuition Breaks"): keys are grouped per
 *     channel (G consecutive tokens of one channel), values per token
 *     (G consecutive channels of one token).  Both axes are selectable, for the
 *     flipped arms of the ablation.
 *   - The full-precision residual (section "The Systems Tax, and Why It Is Not a
 *     Detail"): tokens that do not yet fill a key group stay in an fp16 tail;
 *     a full tail of G tokens is quantized as one block.  Optionally the tail
 *     also keeps a window of the `residual` most recent tokens in fp16 (a
 *     group is quantized only when it leaves at least `residual` newer tokens
 *     behind), and the first `n_sink` tokens (attention sinks) stay in fp16
 *     for good (section "Where the Work Is Headed": high-precision windows for
 *     recent tokens and for sink tokens).
 *   - Keys quantized before RoPE, RoPE applied after dequantization (section
 *     "Rotary Embeddings Complicate the Keys").
 *   - Attention as the softmax-weighted sum of value vectors (section "Values:
 *     Where the Intuition Breaks").
 *
 * Arithmetic, exactly:
 *   mn, mx  = min and max of the group's fp16 values (converted exactly to fp32)
 *   step32  = (mx - mn) / (2^B - 1)            fp32 subtract, IEEE fp32 divide
 *   scale   = fp16(step32), round to nearest even
 *   zero    = fp16(mn + 0.0f)                  exact; a -0 minimum is stored as +0
 *   code    = 0 for every element if scale == 0, else
 *             clamp(rintf((x - mn) / float(scale)), 0, 2^B - 1)   (half-even)
 *   x_hat   = fmaf(code, float(scale), float(zero))               (fp32)
 * FP8 cache (kvq_config.fp8 = 1; "Rotate, Then Round: The Geometry of
 * KV-Cache Compression", "Key takeaway": FP8 first), same groups:
 *   amax    = max |x| over the group
 *   scale   = fp16(amax / 448)                 IEEE fp32 divide, round to even
 *   zero    = +0
 *   code    = 0 if scale == 0, else E4M3(x / float(scale)): the OCP E4M3
 *             value nearest to the IEEE fp32 quotient, ties to the even
 *             mantissa, saturating at +-448 (bit layout s.eeee.mmm, bias 7)
 *   x_hat   = fmaf(E4M3 value of code, float(scale), float(zero))  (exact)
 * Inputs must be finite fp16; non-finite inputs give unspecified codes.
 *
 * Conventions for every call.
 *   - All device pointers are raw CUDA device addresses, 16-byte aligned,
 *     owned by the caller, and must stay valid until the stream reaches the
 *     work enqueued on them.  Host pointers are plain host memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call that launches work is asynchronous on that stream
 *     and never synchronizes, except kvq_check_device_error.
 *   - Lengths are tracked on the host: every (batch, kv-head) pair holds the
 *     same number of tokens.
 *   - Errors are returned as kvq_status; nothing is thrown across the ABI.  A
 *     call that returns an error other than KVQ_ERR_CUDA leaves the cache
 *     state unchanged.
 *   - Kernels never trap.  A bounded wait that runs out sets a device error
 *     word that kvq_check_device_error reports as KVQ_ERR_DEVICE_CHECK.
 *
 * Device layout of the packed cache (P = batch * n_kv_heads pairs,
 * pair p = b * n_kv_heads + h; NB = max_ctx / G blocks per pair; D = head_dim;
 * bk, bv = bits of K and V; words are little-endian uint32):
 *
 *   block (p, i) starts at byte (p * NB + i) * block_bytes, where
 *   block_bytes = G*D*(bk+bv)/8 + 8*D + 8*n (n = n_outliers), and holds
 *   tokens [i*G, (i+1)*G):
 *     [off_kc, +G*D*bk/8)  K codes, in the side's code order (below).
 *     [off_km, +4*D)       K metadata: D entries {fp16 scale, fp16 zero}
 *                          (scale at the lower address).  Channel axis:
 *                          entry d is channel d's group.  Token axis: entry
 *                          j*(D/G) + g is token j, channels [g*G, (g+1)*G).
 *     [off_ko, +4*n)       K outliers: n uint32 entries, the kept fp16 value
 *                          in bits 0-15 and its position j*D + d in the block
 *                          in bits 16-31, ascending by position.
 *     [off_vc, +G*D*bv/8)  V codes, in the side's code order (below).
 *     [off_vm, +4*D)       V metadata, indexed as for K by V's axis.
 *     [off_vo, +4*n)       V outliers, as for K.
 *   off_kc = 0, off_km = G*D*bk/8, off_ko = off_km + 4*D,
 *   off_vc = off_ko + 4*n, off_vm = off_vc + G*D*bv/8, off_vo = off_vm + 4*D.
 *
 *   Outliers (dense-and-sparse isolation, n > 0; KVQuant's "isolating a small
 *   fraction of outliers", "Why KV Cache Geometry Matters More Than Bit
 *   Precision", section "KV Cache Size, GPU Memory Efficiency, and the Shift
 *   to Geometry-Aware Quantization"): in every block and side the n elements
 *   of largest magnitude (ties: lower position j*D + d) are kept exactly;
 *   every group takes its min and max over its other elements (scale 0 and
 *   zero +0 when none remain); kept positions hold code 0 and dequantize to
 *   their kept value.
 *
 *   Code order of a side (kvq_buffers.code_order_k / code_order_v):
 *   FRAGMENT order when keys are grouped per channel, values per token,
 *   G = 32 and D is 64 or 128 (2, 4 or 8 bits, FP8 included); SEQUENTIAL
 *   order otherwise.
 *     Sequential.  K: token-major, token j's row is D*bk/32 words; channel d
 *       sits in word d/(32/bk) at bit (d % (32/bk))*bk.  V: 32-token chunks
 *       c = j/32; inside a chunk, channel-major: channel d owns bv words at
 *       word offset (c*D + d)*bv; token j sits in word (j%32)/(32/bv) of them
 *       at bit ((j%32) % (32/bv))*bv.
 *     Fragment (the operand order of the decode kernel's fp16 tensor-core
 *       tiles, so that each warp lane turns its own words into operand
 *       registers with masks alone).  The side's codes of a block form a tile
 *       of rows x cols codes: K rows = the 32 tokens, cols = the D channels;
 *       V rows = the D channels, cols = the 32 tokens.  Write
 *         row = 16*mt + 8*hr + g            (g < 8, hr < 2)
 *         col = 16*ks + 8*kh + 2*t + e      (t < 4, e < 2, kh < 2)
 *       The code belongs to lane l = 4*g + t, in that lane's word
 *         w = mt*(cols/32) + ks/2  at bit 16*e + F2[hr][2*(ks%2) + kh]  (2 bits)
 *         w = mt*(cols/16) + ks    at bit 16*e + 8*kh + 4*hr            (4 bits)
 *         w = 2*(mt*(cols/16) + ks) + kh   at bit 8*(2*hr + e)          (8 bits)
 *       with F2[0] = {0, 10, 12, 14}, F2[1] = {2, 4, 6, 8}; word w of lane l
 *       is word ((w/4)*32 + l)*4 + w%4 of the region.
 *
 *   Token order of a pair: T_sink sink tokens, then T_q quantized tokens,
 *   then T_tail tail tokens (positions 0 .. T_sink + T_q + T_tail - 1, used
 *   for RoPE).  Block (p, i) holds quantized tokens [i*G, (i+1)*G), i.e.
 *   positions T_sink + i*G onwards (T_sink = n_sink whenever T_q > 0).
 *
 *   The sink window is fp16 [P][n_sink][D] for K and for V, rows [0, T_sink)
 *   valid.  The tail is fp16 [P][residual + G][D] for K and for V
 *   (kvq_buffers.tail_rows rows per pair), rows [0, T_tail) valid.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,  /* null handle/pointer, misaligned pointer, bad size */
  KVQ_ERR_UNSUPPORTED = 2,  /* a valid config this build has no kernel for     */
  KVQ_ERR_CAPACITY = 3,     /* T_sink + T_q + T_tail + n would exceed max_ctx   */
  KVQ_ERR_OOM = 4,          /* device allocation failed                         */
  KVQ_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed             */
  KVQ_ERR_DEVICE_CHECK = 6  /* a kernel reported a bounded wait that ran out    */
} kvq_status;

typedef enum {
  KVQ_AXIS_CHANNEL = 0, /* group = G consecutive tokens of one channel */
  KVQ_AXIS_TOKEN = 1    /* group = G consecutive channels of one token */
} kvq_axis;

typedef struct {
  int batch;         /* >= 1                                                  */
  int n_q_heads;     /* multiple of n_kv_heads; ratio in {1, 2, 4, 8}          */
  int n_kv_heads;    /* >= 1                                                  */
  int head_dim;      /* 64 or 128                                             */
  int max_ctx;       /* capacity in tokens per pair, >= 1                     */
  int bits_k;        /* 2, 4 or 8                                             */
  int bits_v;        /* 2, 4 or 8                                             */
  int group;         /* G: 32, 64 or 128; head_dim % G == 0 if an axis is TOKEN */
  int axis_k;        /* kvq_axis; the pages' choice is KVQ_AXIS_CHANNEL        */
  int axis_v;        /* kvq_axis; the pages' choice is KVQ_AXIS_TOKEN          */
  int keys_pre_rope; /* 1: keys are stored before RoPE; decode rotates them    */
  float rope_base;   /* RoPE base (e.g. 10000), used when keys_pre_rope = 1    */
  int n_sink;        /* first tokens kept in fp16, never quantized; 0..1024   */
  int residual;      /* most recent tokens kept in fp16 beyond the partial
                        group; 0..4096 (0: the tail holds < G tokens)         */
  int fp8;           /* 1: FP8 cache (requires bits_k = bits_v = 8): codes are
                        E4M3, scale = fp16(max|x| / 448), zero = 0            */
  int n_outliers;    /* dense-and-sparse isolation: elements of largest
                        magnitude kept in fp16 per block and side; 0..64, a
                        multiple of 4.  Nonzero needs keys per channel, values
                        per token, G = 32, 2- or 4-bit sides, no FP8 and keys
                        stored after RoPE (KVQ_ERR_UNSUPPORTED otherwise)    */
} kvq_config;

typedef struct kvq_cache kvq_cache; /* opaque */

/* Device addresses and geometry of a cache, for tests and for callers that
 * read the packed bytes.  All pointers are owned by the cache. */
typedef struct {
  void* blocks;                /* [P][NB][block_bytes] packed blocks            */
  void* k_tail;                /* active K tail, fp16 [P][tail_rows][D]         */
  void* v_tail;                /* active V tail, fp16 [P][tail_rows][D]         */
  size_t block_bytes;
  size_t off_kc, off_km, off_vc, off_vm;
  int blocks_per_pair;         /* NB                                            */
  int n_pairs;                 /* P                                             */
  int T_q;                     /* quantized tokens per pair (multiple of G)     */
  int T_tail;                  /* tail tokens per pair, < residual + G          */
  int code_order_k;            /* 0 sequential, 1 fragment (see the layout)     */
  int code_order_v;
  void* k_sink;                /* K sink window, fp16 [P][n_sink][D]; NULL if n_sink = 0 */
  void* v_sink;                /* V sink window, same                           */
  int T_sink;                  /* sink tokens per pair, <= n_sink               */
  int tail_rows;               /* rows per pair of each tail buffer (residual + G) */
  void* k_tail_buffer[2];      /* the two K tail buffers (kvq_get_row_state says  */
  void* v_tail_buffer[2];      /*   which one holds a row's tail)               */
  int ragged;                  /* 1: rows hold different lengths; the T_* fields
                                  and k_tail / v_tail above describe row 0      */
  size_t off_ko, off_vo;       /* K and V outlier sections (n_outliers entries) */
  int n_outliers;
} kvq_buffers;

/* Validates a config on the host (no GPU needed).  Returns KVQ_OK,
 * KVQ_ERR_INVALID_ARG (malformed) or KVQ_ERR_UNSUPPORTED. */
KVQ_API kvq_status kvq_config_check(const kvq_config* cfg);

/* Device bytes kvq_create allocates for `cfg` (packed blocks, two tail
 * buffers, RoPE table, split workspace, error word).  Host only. */
KVQ_API kvq_status kvq_cache_bytes(const kvq_config* cfg, size_t* bytes);

/* Allocates an empty cache on the current CUDA device and builds its RoPE
 * cos/sin table (fp64 on the host, stored fp32).  *out receives the handle;
 * on error *out is set to NULL and nothing stays allocated. */
KVQ_API kvq_status kvq_create(const kvq_config* cfg, kvq_cache** out);

/* Frees everything the cache owns.  Synchronizes the device first.  NULL is
 * accepted and ignored. */
KVQ_API kvq_status kvq_destroy(kvq_cache* cache);

/* Prefill: resets the cache, then stores every pair's T tokens: the first
 * min(T, n_sink) in the sink window; of the rest (T' tokens), the first
 * T_q = floor((T' - residual) / G) * G (0 if T' < residual) are quantized into
 * blocks and the remaining T' - T_q go to the tail.  With n_sink = residual =
 * 0: tokens [0, floor(T/G)*G) are quantized and T mod G stay in the tail.
 * k, v: device fp16 [batch][n_kv_heads][T][head_dim], contiguous.
 * T = 0 empties the cache.  T > max_ctx -> KVQ_ERR_CAPACITY. */
KVQ_API kvq_status kvq_quantize_prefill(kvq_cache* cache, const void* k,
                                        const void* v, int T, void* stream);

/* Prefill of a batch whose rows hold different numbers of tokens (ragged
 * lengths, a serving batch): resets the cache, then stores lengths[b] tokens
 * into every pair of row b exactly as kvq_quantize_prefill does for one
 * length.  k, v: device fp16 [batch][n_kv_heads][T_stride][head_dim]; row b
 * reads tokens [0, lengths[b]) of its pairs.  lengths: host int [batch], each
 * in [1, T_stride] (KVQ_ERR_INVALID_ARG otherwise; > max_ctx ->
 * KVQ_ERR_CAPACITY).  A ragged cache needs batch <= 64 (KVQ_ERR_UNSUPPORTED
 * otherwise); equal lengths give a uniform cache.  Decode, append and
 * append-decode then work per row; kvq_dequantize and kvq_get_state return
 * KVQ_ERR_UNSUPPORTED for a ragged cache (kvq_get_row_state reports lengths). */
KVQ_API kvq_status kvq_quantize_prefill_ragged(kvq_cache* cache, const void* k,
                                               const void* v, const int* lengths,
                                               int T_stride, void* stream);

/* Decode-time append of n tokens per pair.  New tokens first fill the sink
 * window (while T_sink < n_sink); the others join the tail, which with them
 * forms one sequence: while it holds at least residual + G tokens, its oldest
 * G are quantized into the next block (the tail flush); the rest becomes the
 * new tail.  The result equals a prefill of all tokens at once.
 * k, v: device fp16 [batch][n_kv_heads][n][head_dim], contiguous.  n = 0 is a
 * no-op.  T_sink + T_q + T_tail + n > max_ctx -> KVQ_ERR_CAPACITY. */
KVQ_API kvq_status kvq_append(kvq_cache* cache, const void* k, const void* v,
                              int n, void* stream);

/* Append of n_rows[b] tokens to every pair of row b (0 allowed: the row
 * does not advance).  k, v: device fp16 [batch][n_kv_heads][n_stride][head_dim];
 * n_rows: host int [batch], each in [0, n_stride].  Rows follow kvq_append's
 * rules one by one; unequal counts make the cache ragged (batch <= 64,
 * KVQ_ERR_UNSUPPORTED otherwise).  KVQ_ERR_CAPACITY when a row would exceed
 * max_ctx. */
KVQ_API kvq_status kvq_append_ragged(kvq_cache* cache, const void* k, const void* v,
                                     const int* n_rows, int n_stride, void* stream);

/* Split-K decode attention of one query token per head over every cached
 * token (T_sink fp16 sink tokens, T_q dequantized tokens, T_tail fp16 tail
 * tokens; key t below is the token at position t):
 *   out[b][hq] = sum_t softmax_t(scale * q[b][hq] . k_t) * v_t
 * with query head hq reading kv head hq / (n_q_heads / n_kv_heads).  When
 * keys_pre_rope = 1, key t is rotated (rotate-half RoPE, angle
 * t * base^(-2i/D) on channel pair (i, i + D/2)) after dequantization; q is
 * taken as already rotated.
 * q: device fp16 [batch][n_q_heads][head_dim]; out: device fp32, same shape.
 * An empty cache writes zeros. */
KVQ_API kvq_status kvq_decode_attention(kvq_cache* cache, const void* q,
                                        void* out, float softmax_scale,
                                        void* stream);

/* One decode step: kvq_append(cache, k, v, n) then kvq_decode_attention
 * (cache, q, out), with the same results and errors.  When the appended
 * tokens cause no flush (T_tail + n < residual + G) and go to the tail only
 * (T_sink = n_sink), and the cache uses the
 * tensor-core kernel (keys per channel, values per token, G = 32), both run
 * as one launch: the decode reads the new tokens straight from k and v and
 * stores them into the tail.  Otherwise the append (with its flush) and the
 * decode are enqueued one after the other.  The fp16 tail is the pages'
 * full-precision residual ("Your KV cache doesn't have a bit problem, it has
 * a geometry problem", section "The Systems Tax, and Why It Is Not a
 * Detail").  k, v as for kvq_append (may be NULL when n = 0); q, out as for
 * kvq_decode_attention. */
KVQ_API kvq_status kvq_append_decode(kvq_cache* cache, const void* k,
                                     const void* v, int n, const void* q,
                                     void* out, float softmax_scale,
                                     void* stream);

/* Dequantizes the T_q packed tokens of every pair (before any RoPE).
 * k_out, v_out: device fp32 [batch][n_kv_heads][T_q][head_dim]. */
KVQ_API kvq_status kvq_dequantize(kvq_cache* cache, void* k_out, void* v_out,
                                  void* stream);

/* Size of the static device workspace of kvq_decode_attention_noalloc. */
#define KVQ_NOALLOC_SCRATCH_BYTES (8u << 20)

/* Decode attention without allocating device memory (the pages have no
 * counterpart of this call; it exists for callers, not for the method).
 * Some callers cannot call cudaMalloc when they decode: a serving runtime
 * that reserved all device memory in its own arena at start-up, a plugin
 * host that only hands a library the buffers it owns, or a latency-critical
 * loop where an allocation (which can synchronize the device) is not
 * acceptable.  If such a caller holds a packed cache in its own memory, in
 * the layout described at the top of this header, this call decodes it
 * without a kvq_cache (whose creation allocates) and calls no allocating
 * routine.
 *   cfg            the cache's geometry; keys_pre_rope, n_sink, residual
 *                  and n_outliers must be 0 (KVQ_ERR_UNSUPPORTED otherwise:
 *                  the RoPE table would need memory; this call has no window
 *                  buffers and no outlier corrections).
 *   blocks         device, [P][max_ctx/G][block_bytes] packed blocks.
 *   k_tail, v_tail device, fp16 [P][G][D]; rows [0, T_tail) are read.  May be
 *                  NULL when T_tail = 0.
 *   T_q, T_tail    quantized tokens (a multiple of G) and tail tokens
 *                  (< G) per pair; T_q + T_tail <= max_ctx.
 *   q, out, softmax_scale  as for kvq_decode_attention.
 *   device_error   optional device int; receives 0, or nonzero when a
 *                  bounded wait in the kernel ran out.
 * The split-K partials live in a file-scope device array of
 * KVQ_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds until
 * the process exits.  A shape whose partials cannot fit (P * R * (D + 2) * 4
 * bytes plus one slot per decode warp) returns KVQ_ERR_CAPACITY.  The first
 * call on a device looks up the array's device address and the kernels'
 * occupancy, so make that first call before any stream capture.  All calls
 * share the array: calls that overlap on the GPU (different streams, or
 * different host threads) race on it and must be serialized by the caller.
 * Asynchronous on `stream`. */
KVQ_API kvq_status kvq_decode_attention_noalloc(const kvq_config* cfg, const void* blocks,
                                                const void* k_tail, const void* v_tail,
                                                int T_q, int T_tail, const void* q, void* out,
                                                float softmax_scale, int* device_error,
                                                void* stream);

/* Host-side lengths: quantized tokens and tail tokens per pair
 * (KVQ_ERR_UNSUPPORTED for a ragged cache). */
KVQ_API kvq_status kvq_get_state(const kvq_cache* cache, int* T_q,
                                 int* T_tail);

/* Lengths of batch row `row`: sink, quantized and tail tokens of each of its
 * pairs, and which tail buffer (0 or 1 of kvq_buffers.k_tail_buffer) holds
 * the tail rows. */
KVQ_API kvq_status kvq_get_row_state(const kvq_cache* cache, int row, int* T_sink,
                                     int* T_q, int* T_tail, int* tail_buffer);

/* Device addresses and geometry (see the layout above). */
KVQ_API kvq_status kvq_get_buffers(const kvq_cache* cache, kvq_buffers* out);

/* Synchronizes `stream`, reads and clears the device error word.  Returns
 * KVQ_OK, KVQ_ERR_DEVICE_CHECK (a bounded wait ran out) or KVQ_ERR_CUDA. */
KVQ_API kvq_status kvq_check_device_error(kvq_cache* cache, void* stream);

/* Number of kernels this library has launched in this process. */
KVQ_API uint64_t kvq_launch_count(void);

/* Fault-injection hooks for tests of the failure paths (host side; none of
 * them makes a kernel fault or hang).
 *
 * kvq_debug_fail_allocations: after `after` more successful device
 *   allocations, the next n the library makes fail as if the device were out
 *   of memory (kvq_create then returns KVQ_ERR_OOM, frees what it had
 *   allocated and leaves *out NULL).  n = 0 turns the injection off; a
 *   negative argument -> KVQ_ERR_INVALID_ARG.  Process-wide.
 * kvq_debug_set_device_error: synchronizes the device and writes `value`
 *   into the cache's device error word, as a kernel whose bounded wait ran
 *   out would (kvq_check_device_error then reports KVQ_ERR_DEVICE_CHECK and
 *   clears the word).
 * kvq_debug_set_wait_limit: the number of try_wait rounds each main-loop
 *   wait of this cache's decode kernels makes before it gives up (records
 *   the error word, waits with the normal limit for its own copies in flight,
 *   and leaves the launch).  0 gives up at the first wait, so a decode
 *   records the error without writing `out`; limit < 0 restores the normal
 *   limit.  Applies to launches enqueued afterwards. */
KVQ_API kvq_status kvq_debug_fail_allocations(int after, int n);
KVQ_API kvq_status kvq_debug_set_device_error(kvq_cache* cache, int value);
KVQ_API kvq_status kvq_debug_set_wait_limit(kvq_cache* cache, int limit);

/* Static description of a status code. */
KVQ_API const char* kvq_status_string(kvq_status s);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
