// kvq_api.cu — the C ABI of include/kvq.h: validation, ownership of the
// device cache, host-side lengths and kernel launches.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "kvq.h"
#include "kvq_decode.cuh"
#include "kvq_decode_mma.cuh"
#include "kvq_device.cuh"

namespace kvq {
size_t quantize_smem_bytes(int D, int G, int nout);
cudaError_t prepare_quantize();
cudaError_t launch_quantize(const QuantParams& q, cudaStream_t stream);
cudaError_t launch_dequantize(const DequantParams& q, cudaStream_t stream);
cudaError_t launch_merge(const MergeParams& mp, int n_pairs, cudaStream_t stream);
cudaError_t launch_merge2(const Merge2Params& mp, int n_pairs, cudaStream_t stream);
}  // namespace kvq

using namespace kvq;

namespace {

// Most warps a decode launch uses; the partial workspace is sized for it.
constexpr long long kMaxDecodeWarps = 4096;
// Virtual units charged after every pair in the tensor-core kernel's split.
constexpr int kPairCost = 2;

std::atomic<uint64_t> g_launches{0};

// Fault injection (kvq_debug_fail_allocations): after g_alloc_pass more
// successful device allocations, the next g_alloc_fail ones fail as if the
// device were out of memory.
std::mutex g_alloc_mu;
int g_alloc_pass = 0;
int g_alloc_fail = 0;

cudaError_t dev_alloc(void** p, size_t bytes) {
  {
    std::lock_guard<std::mutex> lock(g_alloc_mu);
    if (g_alloc_fail > 0) {
      if (g_alloc_pass > 0) {
        --g_alloc_pass;
      } else {
        --g_alloc_fail;
        *p = nullptr;
        return cudaErrorMemoryAllocation;
      }
    }
  }
  return cudaMalloc(p, bytes);
}

template <typename T>
bool alloc_ok(T** p, size_t bytes) {
  return dev_alloc(reinterpret_cast<void**>(p), bytes) == cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Derived {
  int P, R, NB, G, D;
  int NSK;             // sink window rows per pair (n_sink)
  int residual;        // recent tokens kept in fp16 beyond the partial group
  int TC;              // rows per pair of a tail buffer: residual + G
  int frag_k, frag_v;  // code order of each side (1 fragment, 0 sequential)
  bool mma_geom;       // geometry of the tensor-core decode kernel
  int C2max;  // level-1 chunks per (pair, query) of the two-level merge
  int n_out;           // outliers kept per block and side
  size_t block_bytes, off_kc, off_km, off_ko, off_vc, off_vm, off_vo;
  size_t blocks_bytes, tail_bytes, sink_bytes, rope_bytes, part_o_bytes, part_ml_bytes;
  size_t lvl_o_bytes, lvl_ml_bytes;
};

kvq_status derive(const kvq_config* c, Derived* d) {
  if (c == nullptr) return KVQ_ERR_INVALID_ARG;
  if (c->batch < 1 || c->n_kv_heads < 1 || c->n_q_heads < 1 || c->max_ctx < 1 ||
      c->head_dim < 1 || c->group < 1)
    return KVQ_ERR_INVALID_ARG;
  if (c->n_q_heads % c->n_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  auto bits_ok = [](int b) { return b == 2 || b == 4 || b == 8; };
  if (!bits_ok(c->bits_k) || !bits_ok(c->bits_v)) return KVQ_ERR_INVALID_ARG;
  if ((c->axis_k != 0 && c->axis_k != 1) || (c->axis_v != 0 && c->axis_v != 1))
    return KVQ_ERR_INVALID_ARG;
  if (c->keys_pre_rope != 0 && c->keys_pre_rope != 1) return KVQ_ERR_INVALID_ARG;
  if (c->keys_pre_rope && !(c->rope_base > 1.0f && std::isfinite(c->rope_base)))
    return KVQ_ERR_INVALID_ARG;
  if (c->n_sink < 0 || c->n_sink > 1024 || c->residual < 0 || c->residual > 4096)
    return KVQ_ERR_INVALID_ARG;
  if (c->fp8 != 0 && c->fp8 != 1) return KVQ_ERR_INVALID_ARG;
  if (c->fp8 && (c->bits_k != 8 || c->bits_v != 8)) return KVQ_ERR_INVALID_ARG;
  if (c->n_outliers < 0 || c->n_outliers > 64 || c->n_outliers % 4 != 0) return KVQ_ERR_INVALID_ARG;
  if ((c->axis_k == 1 || c->axis_v == 1) && c->head_dim % c->group != 0)
    return KVQ_ERR_INVALID_ARG;
  const int R = c->n_q_heads / c->n_kv_heads;
  if (R != 1 && R != 2 && R != 4 && R != 8) return KVQ_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (c->group != 32 && c->group != 64 && c->group != 128) return KVQ_ERR_UNSUPPORTED;
  // outlier isolation: the tensor-core geometry with 2- or 4-bit integer
  // sides, keys stored after RoPE
  if (c->n_outliers > 0 &&
      (!mma_geometry(c->group, c->axis_k, c->axis_v) || c->fp8 || c->keys_pre_rope ||
       (c->bits_k != 2 && c->bits_k != 4) || (c->bits_v != 2 && c->bits_v != 4)))
    return KVQ_ERR_UNSUPPORTED;
  const long long P = static_cast<long long>(c->batch) * c->n_kv_heads;
  if (P > 65535) return KVQ_ERR_UNSUPPORTED;  // grid.y of the quantize launch
  if (c->max_ctx > (1 << 26)) return KVQ_ERR_UNSUPPORTED;
  // decode units (32-token sub-blocks, tail and sink chunks of at least six
  // tokens) and their split costs (plus kPairCost per pair) are counted in int
  if (P * (static_cast<long long>(c->max_ctx) / 32 + (c->n_sink + c->residual + c->group) / 6 + 2 +
           kPairCost) >= (1LL << 31))
    return KVQ_ERR_UNSUPPORTED;
  d->P = static_cast<int>(P);
  d->R = R;
  d->mma_geom = mma_geometry(c->group, c->axis_k, c->axis_v);
  d->frag_k = fragment_order(c->head_dim, c->group, c->bits_k, c->axis_k, c->axis_v) ? 1 : 0;
  d->frag_v = fragment_order(c->head_dim, c->group, c->bits_v, c->axis_k, c->axis_v) ? 1 : 0;
  d->G = c->group;
  d->D = c->head_dim;
  d->NSK = c->n_sink;
  d->residual = c->residual;
  d->TC = c->residual + c->group;
  d->NB = c->max_ctx / c->group;
  const size_t D = c->head_dim, G = c->group, n = c->n_outliers;
  d->n_out = c->n_outliers;
  d->off_kc = 0;
  d->off_km = G * D * c->bits_k / 8;
  d->off_ko = d->off_km + 4 * D;
  d->off_vc = d->off_ko + 4 * n;
  d->off_vm = d->off_vc + G * D * c->bits_v / 8;
  d->off_vo = d->off_vm + 4 * D;
  d->block_bytes = d->off_vo + 4 * n;
  d->blocks_bytes = static_cast<size_t>(P) * d->NB * d->block_bytes;
  d->tail_bytes = static_cast<size_t>(P) * d->TC * D * 2;  // one fp16 [P][TC][D] buffer
  d->sink_bytes = static_cast<size_t>(P) * d->NSK * D * 2;  // one fp16 [P][NSK][D] buffer
  d->rope_bytes = c->keys_pre_rope ? static_cast<size_t>(c->max_ctx) * (D / 2) * sizeof(float2) : 0;
  const size_t slots = static_cast<size_t>(kMaxDecodeWarps + P);
  d->part_o_bytes = slots * R * D * sizeof(float);
  d->part_ml_bytes = slots * R * sizeof(float2);
  d->C2max = static_cast<int>((kMaxDecodeWarps / P + 2 + 15) / 16);
  const size_t lvl = static_cast<size_t>(P) * R * d->C2max;
  d->lvl_o_bytes = lvl * D * sizeof(float);
  d->lvl_ml_bytes = lvl * sizeof(float2);
  return KVQ_OK;
}

struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
      ok = false;
      return;
    }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

}  // namespace

struct kvq_cache {
  kvq_config cfg;
  Derived dv;
  int device;
  int sm_count;
  int decode_warps_per_sm;  // resident warps of the decode kernel per SM
  DecodeOps ops;
  uint8_t* blocks;
  __half* ktail[2];
  __half* vtail[2];
  __half* ksink;  // sink window [P][NSK][D], nullptr when n_sink = 0
  __half* vsink;
  float2* rope;
  float* part_o;
  float2* part_ml;
  int* err;
  int* tickets;  // [P] fused-merge counters, zero between launches
  float* lvl_o;  // two-level merge: level-2 partials
  float2* lvl_ml;
  int* tickets2; // [P*R] two-level merge counters, zero between launches
  bool mma;      // decode runs the tensor-core kernel (which can merge in place)
  uint32_t wait_limit;  // try_wait rounds of a decode kernel's bounded waits
  // Token counts per batch row: sink, quantized, tail, and the row's active
  // tail buffer.  A uniform cache keeps every entry equal to row 0; a ragged
  // cache (rows of different lengths, batch <= kMaxRows) one entry per row.
  bool ragged;
  int T_s[kMaxRows], T_q[kMaxRows], T_t[kMaxRows], act[kMaxRows];
};

// Row records a launch describes: every row of a ragged cache, row 0 of a
// uniform one.
static int row_records(const kvq_cache* c) { return c->ragged ? c->cfg.batch : 1; }

// A uniform cache mirrors row 0 into every record.
static void sync_uniform(kvq_cache* c) {
  if (c->ragged) return;
  for (int b = 1; b < kMaxRows; ++b) {
    c->T_s[b] = c->T_s[0];
    c->T_q[b] = c->T_q[0];
    c->T_t[b] = c->T_t[0];
    c->act[b] = c->act[0];
  }
}

static void reset_lengths(kvq_cache* c) {
  c->ragged = false;
  for (int b = 0; b < kMaxRows; ++b) c->T_s[b] = c->T_q[b] = c->T_t[b] = c->act[b] = 0;
}

// Tokens of row b.
static long long row_tokens(const kvq_cache* c, int b) {
  return static_cast<long long>(c->T_s[b]) + c->T_q[b] + c->T_t[b];
}

static CacheGeom geom_of(const kvq_cache* c) {
  CacheGeom g;
  g.blocks = c->blocks;
  g.block_bytes = c->dv.block_bytes;
  g.NB = c->dv.NB;
  g.off_km = static_cast<int>(c->dv.off_km);
  g.off_vc = static_cast<int>(c->dv.off_vc);
  g.off_vm = static_cast<int>(c->dv.off_vm);
  g.D = c->dv.D;
  g.G = c->dv.G;
  g.frag_k = c->dv.frag_k;
  g.frag_v = c->dv.frag_v;
  g.bk = c->cfg.bits_k;
  g.bv = c->cfg.bits_v;
  g.ak = c->cfg.axis_k;
  g.av = c->cfg.axis_v;
  g.P = c->dv.P;
  g.fp8 = c->cfg.fp8;
  g.TC = c->dv.TC;
  g.NSK = c->dv.NSK;
  g.nout = c->dv.n_out;
  g.off_ko = static_cast<int>(c->dv.off_ko);
  g.off_vo = static_cast<int>(c->dv.off_vo);
  return g;
}

static void free_all(kvq_cache* c) {
  cudaFree(c->blocks);
  for (int i = 0; i < 2; ++i) {
    cudaFree(c->ktail[i]);
    cudaFree(c->vtail[i]);
  }
  cudaFree(c->ksink);
  cudaFree(c->vsink);
  cudaFree(c->rope);
  cudaFree(c->part_o);
  cudaFree(c->part_ml);
  cudaFree(c->err);
  cudaFree(c->tickets);
  cudaFree(c->lvl_o);
  cudaFree(c->lvl_ml);
  cudaFree(c->tickets2);
}

// Appends to every pair of row b its n_rows[b] tokens (n_all for every row
// when n_rows is null); k, v: [P][stride][D].  The first tokens of a row fill
// its sink window while it is short, the others join the tail; every group of
// G that leaves at least `residual` newer tail tokens is quantized.  The whole
// combined tail + new sequence is walked once (see QuantParams).
static kvq_status enqueue_append(kvq_cache* c, const void* k, const void* v, const int* n_rows,
                                 int n_all, int stride, cudaStream_t stream) {
  const int G = c->dv.G;
  const int nr = row_records(c);
  QuantParams q;
  q.g = geom_of(c);
  q.knew = static_cast<const __half*>(k);
  q.vnew = static_cast<const __half*>(v);
  q.new_stride = stride;
  for (int i = 0; i < 2; ++i) {
    q.ktail[i] = c->ktail[i];
    q.vtail[i] = c->vtail[i];
  }
  q.ksink = c->ksink;
  q.vsink = c->vsink;
  q.ragged = c->ragged ? 1 : 0;
  q.hkv = c->cfg.n_kv_heads;
  bool any = false;
  for (int b = 0; b < nr; ++b) {
    QuantRow& r = q.rows[b];
    r.n = n_rows ? n_rows[b] : n_all;
    r.sink0 = c->T_s[b];
    r.nsink = std::min(r.n, c->dv.NSK - c->T_s[b]);
    const int combined = c->T_t[b] + (r.n - r.nsink);
    r.nflush = combined >= c->dv.residual ? (combined - c->dv.residual) / G : 0;
    r.T_t = c->T_t[b];
    r.src = c->act[b];
    r.first_block = c->T_q[b] / G;
    if (r.nflush == 0) {
      r.dst = r.src;
      r.dst_row0 = c->T_t[b];
      r.rem_begin = c->T_t[b];
    } else {  // the flush reads the old tail: the remainder goes to the other buffer
      r.dst = r.src ^ 1;
      r.dst_row0 = 0;
      r.rem_begin = r.nflush * G;
    }
    r.rem_end = combined;
    any = any || r.n > 0;
  }
  if (!any) return KVQ_OK;
  if (launch_quantize(q, stream) != cudaSuccess) return KVQ_ERR_CUDA;
  g_launches.fetch_add(1);
  for (int b = 0; b < nr; ++b) {
    const QuantRow& r = q.rows[b];
    c->T_s[b] += r.nsink;
    c->T_q[b] += r.nflush * G;
    c->T_t[b] = r.rem_end - r.nflush * G;
    c->act[b] = r.dst;
  }
  sync_uniform(c);
  return KVQ_OK;
}

extern "C" {

kvq_status kvq_config_check(const kvq_config* cfg) {
  Derived d;
  return derive(cfg, &d);
}

kvq_status kvq_cache_bytes(const kvq_config* cfg, size_t* bytes) {
  if (bytes == nullptr) return KVQ_ERR_INVALID_ARG;
  Derived d;
  kvq_status s = derive(cfg, &d);
  if (s != KVQ_OK) return s;
  *bytes = d.blocks_bytes + 4 * d.tail_bytes + 2 * d.sink_bytes + d.rope_bytes + d.part_o_bytes +
           d.part_ml_bytes + d.lvl_o_bytes + d.lvl_ml_bytes + sizeof(int) +
           sizeof(int) * static_cast<size_t>(d.P) * (1 + d.R);
  return KVQ_OK;
}

kvq_status kvq_create(const kvq_config* cfg, kvq_cache** out) {
  if (out == nullptr) return KVQ_ERR_INVALID_ARG;
  *out = nullptr;
  Derived d;
  kvq_status s = derive(cfg, &d);
  if (s != KVQ_OK) return s;
  // Tensor-core kernel for channel-grouped keys, token-grouped values and
  // G = 32 (with its rotated-key variant for keys stored before RoPE); the
  // CUDA-core kernel for every other geometry.  Codes in fragment order are
  // read by the tensor-core kernel only.
  // (an FP8 cache dispatches on the E4M3 tag instead of its 8 bits)
  const int bk = cfg->fp8 ? kBitsE4M3 : cfg->bits_k, bv = cfg->fp8 ? kBitsE4M3 : cfg->bits_v;
  DecodeOps ops{nullptr, nullptr};
  if (d.mma_geom) ops = decode_mma_ops(d.D, d.R, bk, bv, cfg->keys_pre_rope != 0, d.n_out > 0);
  const bool mma = ops.launch != nullptr;
  if ((d.frag_k || d.frag_v) && !mma) return KVQ_ERR_UNSUPPORTED;
  if (ops.launch == nullptr) ops = decode_ops(d.D, d.R, bk, bv);
  if (ops.launch == nullptr) return KVQ_ERR_UNSUPPORTED;

  kvq_cache* c = new (std::nothrow) kvq_cache();
  if (c == nullptr) return KVQ_ERR_OOM;
  c->cfg = *cfg;
  c->dv = d;
  c->ops = ops;
  c->mma = mma;
  c->wait_limit = kWaitLimit;
  if (cudaGetDevice(&c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, c->device) !=
          cudaSuccess ||
      ops.prepare(&c->decode_warps_per_sm) != cudaSuccess || prepare_quantize() != cudaSuccess) {
    cudaGetLastError();
    delete c;
    return KVQ_ERR_CUDA;
  }
  if (c->decode_warps_per_sm < 1) {
    delete c;
    return KVQ_ERR_UNSUPPORTED;
  }
  bool ok = alloc_ok(&c->blocks, d.blocks_bytes > 0 ? d.blocks_bytes : 16);
  for (int i = 0; i < 2 && ok; ++i)
    ok = alloc_ok(&c->ktail[i], d.tail_bytes) && alloc_ok(&c->vtail[i], d.tail_bytes);
  if (ok && d.sink_bytes) ok = alloc_ok(&c->ksink, d.sink_bytes) && alloc_ok(&c->vsink, d.sink_bytes);
  if (ok && d.rope_bytes) ok = alloc_ok(&c->rope, d.rope_bytes);
  if (ok) ok = alloc_ok(&c->part_o, d.part_o_bytes);
  if (ok) ok = alloc_ok(&c->part_ml, d.part_ml_bytes);
  if (ok) ok = alloc_ok(&c->err, sizeof(int));
  if (ok) ok = alloc_ok(&c->tickets, sizeof(int) * d.P);
  if (ok) ok = alloc_ok(&c->lvl_o, d.lvl_o_bytes);
  if (ok) ok = alloc_ok(&c->lvl_ml, d.lvl_ml_bytes);
  if (ok) ok = alloc_ok(&c->tickets2, sizeof(int) * d.P * d.R);
  if (!ok) {
    cudaGetLastError();
    free_all(c);
    delete c;
    return KVQ_ERR_OOM;
  }
  bool init_ok = cudaMemset(c->err, 0, sizeof(int)) == cudaSuccess &&
                 cudaMemset(c->tickets, 0, sizeof(int) * d.P) == cudaSuccess &&
                 cudaMemset(c->tickets2, 0, sizeof(int) * d.P * d.R) == cudaSuccess;
  for (int i = 0; i < 2 && init_ok; ++i)
    init_ok = cudaMemset(c->ktail[i], 0, d.tail_bytes) == cudaSuccess &&
              cudaMemset(c->vtail[i], 0, d.tail_bytes) == cudaSuccess;
  if (init_ok && d.sink_bytes)
    init_ok = cudaMemset(c->ksink, 0, d.sink_bytes) == cudaSuccess &&
              cudaMemset(c->vsink, 0, d.sink_bytes) == cudaSuccess;
  if (init_ok && d.rope_bytes) {
    // RoPE cos/sin table: angle pos * base^(-2i/D), evaluated in fp64.
    const int half = d.D / 2;
    std::vector<float2> tab(static_cast<size_t>(cfg->max_ctx) * half);
    for (int i = 0; i < half; ++i) {
      const double theta = std::pow(static_cast<double>(cfg->rope_base),
                                    -2.0 * static_cast<double>(i) / static_cast<double>(d.D));
      for (int pos = 0; pos < cfg->max_ctx; ++pos) {
        const double a = static_cast<double>(pos) * theta;
        tab[static_cast<size_t>(pos) * half + i] =
            make_float2(static_cast<float>(std::cos(a)), static_cast<float>(std::sin(a)));
      }
    }
    init_ok = cudaMemcpy(c->rope, tab.data(), d.rope_bytes, cudaMemcpyHostToDevice) == cudaSuccess;
  }
  if (!init_ok) {
    cudaGetLastError();
    free_all(c);
    delete c;
    return KVQ_ERR_CUDA;
  }
  *out = c;
  return KVQ_OK;
}

kvq_status kvq_destroy(kvq_cache* c) {
  if (c == nullptr) return KVQ_OK;
  DeviceGuard g(c->device);
  cudaDeviceSynchronize();
  free_all(c);
  delete c;
  return KVQ_OK;
}

// Saved host lengths, restored when an enqueue fails before any launch.
struct SavedLengths {
  bool ragged;
  int T_s[kMaxRows], T_q[kMaxRows], T_t[kMaxRows], act[kMaxRows];
  explicit SavedLengths(const kvq_cache* c) : ragged(c->ragged) {
    std::memcpy(T_s, c->T_s, sizeof(T_s));
    std::memcpy(T_q, c->T_q, sizeof(T_q));
    std::memcpy(T_t, c->T_t, sizeof(T_t));
    std::memcpy(act, c->act, sizeof(act));
  }
  void restore(kvq_cache* c) const {
    c->ragged = ragged;
    std::memcpy(c->T_s, T_s, sizeof(T_s));
    std::memcpy(c->T_q, T_q, sizeof(T_q));
    std::memcpy(c->T_t, T_t, sizeof(T_t));
    std::memcpy(c->act, act, sizeof(act));
  }
};

kvq_status kvq_quantize_prefill(kvq_cache* c, const void* k, const void* v, int T,
                                void* stream) {
  if (c == nullptr || T < 0) return KVQ_ERR_INVALID_ARG;
  if (T > 0 && (k == nullptr || v == nullptr || !aligned16(k) || !aligned16(v)))
    return KVQ_ERR_INVALID_ARG;
  if (T > c->cfg.max_ctx) return KVQ_ERR_CAPACITY;
  DeviceGuard g(c->device);
  if (!g.ok) return KVQ_ERR_CUDA;
  const SavedLengths saved(c);
  reset_lengths(c);
  if (T == 0) return KVQ_OK;
  kvq_status s = enqueue_append(c, k, v, nullptr, T, T, static_cast<cudaStream_t>(stream));
  if (s != KVQ_OK) saved.restore(c);
  return s;
}

kvq_status kvq_quantize_prefill_ragged(kvq_cache* c, const void* k, const void* v,
                                       const int* lengths, int T_stride, void* stream) {
  if (c == nullptr || lengths == nullptr || T_stride < 1) return KVQ_ERR_INVALID_ARG;
  if (k == nullptr || v == nullptr || !aligned16(k) || !aligned16(v)) return KVQ_ERR_INVALID_ARG;
  const int B = c->cfg.batch;
  if (B > kMaxRows) return KVQ_ERR_UNSUPPORTED;
  bool same = true;
  for (int b = 0; b < B; ++b) {
    if (lengths[b] < 1 || lengths[b] > T_stride) return KVQ_ERR_INVALID_ARG;
    same = same && lengths[b] == lengths[0];
  }
  for (int b = 0; b < B; ++b)
    if (lengths[b] > c->cfg.max_ctx) return KVQ_ERR_CAPACITY;
  DeviceGuard g(c->device);
  if (!g.ok) return KVQ_ERR_CUDA;
  const SavedLengths saved(c);
  reset_lengths(c);
  c->ragged = !same;
  kvq_status s = same ? enqueue_append(c, k, v, nullptr, lengths[0], T_stride,
                                       static_cast<cudaStream_t>(stream))
                      : enqueue_append(c, k, v, lengths, 0, T_stride,
                                       static_cast<cudaStream_t>(stream));
  if (s != KVQ_OK) saved.restore(c);
  return s;
}

kvq_status kvq_append(kvq_cache* c, const void* k, const void* v, int n, void* stream) {
  if (c == nullptr || n < 0) return KVQ_ERR_INVALID_ARG;
  if (n == 0) return KVQ_OK;
  if (k == nullptr || v == nullptr || !aligned16(k) || !aligned16(v)) return KVQ_ERR_INVALID_ARG;
  for (int b = 0; b < row_records(c); ++b)
    if (row_tokens(c, b) + n > c->cfg.max_ctx) return KVQ_ERR_CAPACITY;
  DeviceGuard g(c->device);
  if (!g.ok) return KVQ_ERR_CUDA;
  return enqueue_append(c, k, v, nullptr, n, n, static_cast<cudaStream_t>(stream));
}

kvq_status kvq_append_ragged(kvq_cache* c, const void* k, const void* v, const int* n_rows,
                             int n_stride, void* stream) {
  if (c == nullptr || n_rows == nullptr || n_stride < 1) return KVQ_ERR_INVALID_ARG;
  const int B = c->cfg.batch;
  if (B > kMaxRows) return KVQ_ERR_UNSUPPORTED;
  bool same = true, any = false;
  for (int b = 0; b < B; ++b) {
    if (n_rows[b] < 0 || n_rows[b] > n_stride) return KVQ_ERR_INVALID_ARG;
    same = same && n_rows[b] == n_rows[0];
    any = any || n_rows[b] > 0;
  }
  if (!any) return KVQ_OK;
  if (k == nullptr || v == nullptr || !aligned16(k) || !aligned16(v)) return KVQ_ERR_INVALID_ARG;
  for (int b = 0; b < B; ++b)
    if (row_tokens(c, c->ragged ? b : 0) + n_rows[b] > c->cfg.max_ctx) return KVQ_ERR_CAPACITY;
  DeviceGuard g(c->device);
  if (!g.ok) return KVQ_ERR_CUDA;
  const SavedLengths saved(c);
  if (!same) c->ragged = true;  // uniform records already mirror row 0
  kvq_status s = enqueue_append(c, k, v, c->ragged ? n_rows : nullptr, n_rows[0], n_stride,
                                static_cast<cudaStream_t>(stream));
  if (s != KVQ_OK) saved.restore(c);
  return s;
}

// Enqueues the decode of the cache's tokens plus, when n_new > 0 (tensor-core
// kernel only, no flush), the n_new tokens of knew/vnew of every pair, which
// the same launch also stores into the tail.  The caller updates the lengths.
static kvq_status enqueue_decode(kvq_cache* c, const void* q, void* out, float softmax_scale,
                                 cudaStream_t st, const void* knew, const void* vnew, int n_new) {
  const Derived& d = c->dv;
  const int nr = row_records(c);
  DecodeParams p;
  UnitMap& m = p.map;
  m.ragged = c->ragged ? 1 : 0;
  m.hkv = c->cfg.n_kv_heads;
  const int tch = c->mma ? mma_tail_chunk(c->cfg.bits_k, c->cfg.bits_v) : 0;
  p.act = 0;
  for (int b = 0; b < nr; ++b) {
    m.Ts[b] = c->T_s[b];
    m.Tq[b] = c->T_q[b];
    m.Tt[b] = c->T_t[b] + n_new;
    set_row_units(m, b, tch);
    if (c->act[b]) p.act |= 1ull << b;
  }
  m.rows = nr;
  int max_upp = 0;
  for (int b = 0; b < nr; ++b) max_upp = std::max(max_upp, units_of_row(m, b));
  long long target = static_cast<long long>(c->sm_count) * c->decode_warps_per_sm;
  if (target > kMaxDecodeWarps) target = kMaxDecodeWarps;
  // Leaving a pair (its partial, the merge, the next pair's query and its
  // fp16 tail units) costs the tensor-core kernel about kPairCost units of
  // block work: the split charges each pair that much extra.
  const long long W = finish_map(m, d.P, c->mma ? kPairCost : 0, target);
  const long long U = m.U;
  if (U == 0) {  // an empty cache (n_new is 0 here)
    if (cudaMemsetAsync(out, 0, static_cast<size_t>(d.P) * d.R * d.D * sizeof(float), st) !=
        cudaSuccess)
      return KVQ_ERR_CUDA;
    return KVQ_OK;
  }

  p.g = geom_of(c);
  for (int i = 0; i < 2; ++i) {
    p.ktail[i] = c->ktail[i];
    p.vtail[i] = c->vtail[i];
  }
  p.ksink = c->ksink;
  p.vsink = c->vsink;
  p.n_new = n_new;
  p.knew = static_cast<const __half*>(knew);
  p.vnew = static_cast<const __half*>(vnew);
  p.lg_G = d.G == 32 ? 5 : (d.G == 64 ? 6 : 7);
  p.lg_sub = p.lg_G - 5;
  p.n_warps = static_cast<int>(W);
  p.rope = c->cfg.keys_pre_rope;
  p.rope_tab = c->rope;
  p.rope_rows = c->cfg.max_ctx;
  p.q = static_cast<const __half*>(q);
  p.qscale = softmax_scale * 1.4426950408889634f;
  p.part_o = c->part_o;
  p.part_ml = c->part_ml;
  p.err = c->err;
  p.wait_limit = c->wait_limit;
  // Merge in place when every pair has few partials; the separate merge
  // kernel otherwise (few pairs over many warps, e.g. one long sequence).
  // A pair's costs touch at most (upp + vcost) * W / C + 2 warps.
  const long long max_seg = static_cast<long long>(max_upp + m.vcost) * W / m.C + 2;
  p.fused = (c->mma && max_seg <= 64) ? 1 : 0;
  p.tickets = c->tickets;
  p.out = static_cast<float*>(out);
  if (c->ops.launch(p, st) != cudaSuccess) return KVQ_ERR_CUDA;
  if (p.fused) {
    g_launches.fetch_add(1);
    return KVQ_OK;
  }
  Merge2Params mp;
  mp.part_o = c->part_o;
  mp.part_ml = c->part_ml;
  mp.lvl_o = c->lvl_o;
  mp.lvl_ml = c->lvl_ml;
  mp.tickets = c->tickets2;
  mp.out = static_cast<float*>(out);
  mp.map = m;
  mp.R = d.R;
  mp.D = d.D;
  // chunks of CS partial slots, at most C2max chunks per (pair, query)
  mp.CS = static_cast<int>(std::max<long long>(16, (max_seg + d.C2max - 1) / d.C2max));
  mp.C2 = static_cast<int>((max_seg + mp.CS - 1) / mp.CS);
  if (mp.CS > kMerge2MaxRows || mp.C2 > kMerge2MaxRows) return KVQ_ERR_UNSUPPORTED;
  if (launch_merge2(mp, d.P, st) != cudaSuccess) return KVQ_ERR_CUDA;
  g_launches.fetch_add(2);
  return KVQ_OK;
}

kvq_status kvq_decode_attention(kvq_cache* c, const void* q, void* out, float softmax_scale,
                                void* stream) {
  if (c == nullptr || q == nullptr || out == nullptr || !aligned16(q) || !aligned16(out))
    return KVQ_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return KVQ_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  if (!g.ok) return KVQ_ERR_CUDA;
  return enqueue_decode(c, q, out, softmax_scale, static_cast<cudaStream_t>(stream), nullptr,
                        nullptr, 0);
}

kvq_status kvq_append_decode(kvq_cache* c, const void* k, const void* v, int n, const void* q,
                             void* out, float softmax_scale, void* stream) {
  if (c == nullptr || n < 0 || q == nullptr || out == nullptr || !aligned16(q) ||
      !aligned16(out))
    return KVQ_ERR_INVALID_ARG;
  if (n > 0 && (k == nullptr || v == nullptr || !aligned16(k) || !aligned16(v)))
    return KVQ_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return KVQ_ERR_INVALID_ARG;
  const int nr = row_records(c);
  for (int b = 0; b < nr; ++b)
    if (row_tokens(c, b) + n > c->cfg.max_ctx) return KVQ_ERR_CAPACITY;
  DeviceGuard g(c->device);
  if (!g.ok) return KVQ_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // one launch when every row's new tokens go to its tail without a flush
  bool fuse = n > 0 && c->mma;
  for (int b = 0; b < nr && fuse; ++b)
    fuse = c->T_s[b] == c->dv.NSK && c->T_t[b] + n < c->dv.residual + c->dv.G;
  if (fuse) {
    const kvq_status s = enqueue_decode(c, q, out, softmax_scale, st, k, v, n);
    if (s == KVQ_OK) {
      for (int b = 0; b < kMaxRows; ++b) c->T_t[b] += n;
    }
    return s;
  }
  if (n > 0) {
    const kvq_status s = enqueue_append(c, k, v, nullptr, n, n, st);
    if (s != KVQ_OK) return s;
  }
  return enqueue_decode(c, q, out, softmax_scale, st, nullptr, nullptr, 0);
}

kvq_status kvq_dequantize(kvq_cache* c, void* k_out, void* v_out, void* stream) {
  if (c == nullptr) return KVQ_ERR_INVALID_ARG;
  if (c->ragged) return KVQ_ERR_UNSUPPORTED;  // rows of different lengths
  if (c->T_q[0] == 0) return KVQ_OK;  // nothing to write; the outputs may be empty
  if (k_out == nullptr || v_out == nullptr || !aligned16(k_out) || !aligned16(v_out))
    return KVQ_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  if (!g.ok) return KVQ_ERR_CUDA;
  DequantParams p;
  p.g = geom_of(c);
  p.T_q = c->T_q[0];
  p.kout = static_cast<float*>(k_out);
  p.vout = static_cast<float*>(v_out);
  if (launch_dequantize(p, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVQ_ERR_CUDA;
  g_launches.fetch_add(1);
  return KVQ_OK;
}

kvq_status kvq_get_state(const kvq_cache* c, int* T_q, int* T_tail) {
  if (c == nullptr || T_q == nullptr || T_tail == nullptr) return KVQ_ERR_INVALID_ARG;
  if (c->ragged) return KVQ_ERR_UNSUPPORTED;
  *T_q = c->T_q[0];
  *T_tail = c->T_t[0];
  return KVQ_OK;
}

kvq_status kvq_get_row_state(const kvq_cache* c, int row, int* T_sink, int* T_q, int* T_tail,
                             int* tail_buffer) {
  if (c == nullptr || row < 0 || row >= c->cfg.batch || T_sink == nullptr || T_q == nullptr ||
      T_tail == nullptr || tail_buffer == nullptr)
    return KVQ_ERR_INVALID_ARG;
  const int b = c->ragged ? row : 0;
  *T_sink = c->T_s[b];
  *T_q = c->T_q[b];
  *T_tail = c->T_t[b];
  *tail_buffer = c->act[b];
  return KVQ_OK;
}

kvq_status kvq_get_buffers(const kvq_cache* c, kvq_buffers* out) {
  if (c == nullptr || out == nullptr) return KVQ_ERR_INVALID_ARG;
  out->blocks = c->blocks;
  out->k_tail = c->ktail[c->act[0]];
  out->v_tail = c->vtail[c->act[0]];
  out->block_bytes = c->dv.block_bytes;
  out->off_kc = c->dv.off_kc;
  out->off_km = c->dv.off_km;
  out->off_vc = c->dv.off_vc;
  out->off_vm = c->dv.off_vm;
  out->code_order_k = c->dv.frag_k;
  out->code_order_v = c->dv.frag_v;
  out->blocks_per_pair = c->dv.NB;
  out->n_pairs = c->dv.P;
  out->T_q = c->T_q[0];
  out->T_tail = c->T_t[0];
  out->k_sink = c->ksink;
  out->v_sink = c->vsink;
  out->T_sink = c->T_s[0];
  out->tail_rows = c->dv.TC;
  for (int i = 0; i < 2; ++i) {
    out->k_tail_buffer[i] = c->ktail[i];
    out->v_tail_buffer[i] = c->vtail[i];
  }
  out->ragged = c->ragged ? 1 : 0;
  out->off_ko = c->dv.off_ko;
  out->off_vo = c->dv.off_vo;
  out->n_outliers = c->dv.n_out;
  return KVQ_OK;
}

kvq_status kvq_check_device_error(kvq_cache* c, void* stream) {
  if (c == nullptr) return KVQ_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  if (!g.ok) return KVQ_ERR_CUDA;
  int h = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess ||
      cudaMemcpy(&h, c->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(c->err, 0, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_ERR_CUDA;
  }
  if (h != 0) {
    // A warp that gave up left its pair's ticket short: start clean.
    cudaMemset(c->tickets, 0, sizeof(int) * c->dv.P);
    cudaMemset(c->tickets2, 0, sizeof(int) * c->dv.P * c->dv.R);
    return KVQ_ERR_DEVICE_CHECK;
  }
  return KVQ_OK;
}

uint64_t kvq_launch_count(void) { return g_launches.load(); }

kvq_status kvq_debug_fail_allocations(int after, int n) {
  if (after < 0 || n < 0) return KVQ_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_alloc_mu);
  g_alloc_pass = after;
  g_alloc_fail = n;
  return KVQ_OK;
}

kvq_status kvq_debug_set_device_error(kvq_cache* c, int value) {
  if (c == nullptr) return KVQ_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  if (!g.ok) return KVQ_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(c->err, &value, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_ERR_CUDA;
  }
  return KVQ_OK;
}

kvq_status kvq_debug_set_wait_limit(kvq_cache* c, int limit) {
  if (c == nullptr) return KVQ_ERR_INVALID_ARG;
  c->wait_limit = limit < 0 ? kWaitLimit : static_cast<uint32_t>(limit);
  return KVQ_OK;
}

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ_ERR_CAPACITY: return "capacity exceeded";
    case KVQ_ERR_OOM: return "device allocation failed";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_DEVICE_CHECK: return "device check failed (a bounded wait ran out)";
  }
  return "unknown status";
}

}  // extern "C"

namespace kvq {
// Lets other translation units of the library count their launches.
void count_launches(uint64_t n) { g_launches.fetch_add(n); }
}  // namespace kvq
