// kvq_noalloc.cu — decode attention that allocates no device memory.
//
// Some callers cannot call cudaMalloc when they need a decode: a serving
// runtime that hands out all device memory from an arena it reserved at
// start-up and forbids allocation afterwards, a plugin host that gives a
// library only the buffers it owns, or a latency-critical loop where an
// allocation (which can synchronize the device) is not acceptable.  If such a
// caller holds a packed cache in its own memory, in the layout of kvq.h, it
// can decode it with kvq_decode_attention_noalloc.  The only device memory
// that entry point needs besides its arguments, the split-K partials and an
// error word, lives in the file-scope array below, which every GPU that loads
// the library holds until the process exits.
//
// The decode and merge kernels are the ones kvq_decode_attention launches;
// only the workspace they write to differs.
#include <cmath>
#include <mutex>

#include "kvq.h"
#include "kvq_decode.cuh"
#include "kvq_decode_mma.cuh"

namespace kvq {
cudaError_t launch_merge(const MergeParams& mp, int n_pairs, cudaStream_t stream);
void count_launches(uint64_t n);
}  // namespace kvq

using namespace kvq;

namespace {

// The static workspace.  In host code `g_noalloc_scratch` is only a symbol,
// not a device address: the address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
constexpr long long kMaxWarps = 4096;

struct DeviceSetup {
  bool done = false;
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch
  int sm_count = 0;
};

std::mutex g_mu;
DeviceSetup g_setup[kMaxDevices];

struct OccEntry {
  int device;
  cudaError_t (*prepare)(int*);
  int warps_per_sm;
};
OccEntry g_occ[256];
int g_n_occ = 0;

// Once per device, with that device current: the scratch address and the SM
// count.  Also the per-kernel shared-memory opt-in and occupancy, once per
// (device, kernel).  None of these calls allocates device memory.
kvq_status setup(int dev, const DecodeOps& ops, DeviceSetup* out, int* warps_per_sm) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (dev < 0 || dev >= kMaxDevices) return KVQ_ERR_UNSUPPORTED;
  DeviceSetup& s = g_setup[dev];
  if (!s.done) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess ||
        cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return KVQ_ERR_CUDA;
    }
    s.scratch = static_cast<unsigned char*>(ptr);
    s.done = true;
  }
  for (int i = 0; i < g_n_occ; ++i) {
    if (g_occ[i].device == dev && g_occ[i].prepare == ops.prepare) {
      *out = s;
      *warps_per_sm = g_occ[i].warps_per_sm;
      return KVQ_OK;
    }
  }
  int n = 0;
  if (ops.prepare(&n) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_ERR_CUDA;
  }
  if (n < 1) return KVQ_ERR_UNSUPPORTED;
  if (g_n_occ < 256) g_occ[g_n_occ++] = OccEntry{dev, ops.prepare, n};
  *out = s;
  *warps_per_sm = n;
  return KVQ_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

extern "C" kvq_status kvq_decode_attention_noalloc(const kvq_config* cfg, const void* blocks,
                                                   const void* k_tail, const void* v_tail,
                                                   int T_q, int T_tail, const void* q, void* out,
                                                   float softmax_scale, int* device_error,
                                                   void* stream) {
  const kvq_status cs = kvq_config_check(cfg);
  if (cs != KVQ_OK) return cs;
  if (cfg->keys_pre_rope) return KVQ_ERR_UNSUPPORTED;  // the RoPE table would need memory
  if (cfg->n_sink != 0 || cfg->residual != 0) return KVQ_ERR_UNSUPPORTED;  // no window buffers
  if (cfg->n_outliers != 0) return KVQ_ERR_UNSUPPORTED;  // its corrections need the cache's kernels
  const int D = cfg->head_dim, G = cfg->group;
  const int R = cfg->n_q_heads / cfg->n_kv_heads;
  const long long P = static_cast<long long>(cfg->batch) * cfg->n_kv_heads;
  const int NB = cfg->max_ctx / G;
  if (T_q < 0 || T_tail < 0 || T_tail >= G || T_q % G != 0 ||
      static_cast<long long>(T_q) + T_tail > cfg->max_ctx || T_q / G > NB)
    return KVQ_ERR_INVALID_ARG;
  if (blocks == nullptr || q == nullptr || out == nullptr || !aligned16(blocks) ||
      !aligned16(q) || !aligned16(out))
    return KVQ_ERR_INVALID_ARG;
  if (T_tail > 0 && (k_tail == nullptr || v_tail == nullptr || !aligned16(k_tail) ||
                     !aligned16(v_tail)))
    return KVQ_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return KVQ_ERR_INVALID_ARG;

  // Scratch layout: partial outputs [slots][R][D] fp32, partial (m, l)
  // [slots][R] float2, one error word.  slots = warps + pairs.
  const size_t slot_o = static_cast<size_t>(R) * D * sizeof(float);
  const size_t slot_ml = static_cast<size_t>(R) * sizeof(float2);
  const size_t fixed = 2 * 256 + sizeof(int);
  if (KVQ_NOALLOC_SCRATCH_BYTES < fixed ||
      (KVQ_NOALLOC_SCRATCH_BYTES - fixed) / (slot_o + slot_ml) < static_cast<size_t>(P) + 1)
    return KVQ_ERR_CAPACITY;  // the pairs' partials do not fit in the static workspace
  const long long max_slots =
      static_cast<long long>((KVQ_NOALLOC_SCRATCH_BYTES - fixed) / (slot_o + slot_ml));

  const int bk = cfg->fp8 ? kBitsE4M3 : cfg->bits_k, bv = cfg->fp8 ? kBitsE4M3 : cfg->bits_v;
  DecodeOps ops{nullptr, nullptr};
  if (mma_geometry(G, cfg->axis_k, cfg->axis_v))
    ops = decode_mma_ops(D, R, bk, bv, false);
  const bool mma = ops.launch != nullptr;
  if (!mma && (fragment_order(D, G, cfg->bits_k, cfg->axis_k, cfg->axis_v) ||
               fragment_order(D, G, cfg->bits_v, cfg->axis_k, cfg->axis_v)))
    return KVQ_ERR_UNSUPPORTED;
  if (ops.launch == nullptr) ops = decode_ops(D, R, bk, bv);
  if (ops.launch == nullptr) return KVQ_ERR_UNSUPPORTED;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_ERR_CUDA;
  }
  DeviceSetup ds;
  int warps_per_sm = 0;
  const kvq_status ss = setup(dev, ops, &ds, &warps_per_sm);
  if (ss != KVQ_OK) return ss;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  UnitMap map;
  map.ragged = 0;
  map.hkv = cfg->n_kv_heads;
  map.rows = 1;
  map.Ts[0] = 0;
  map.Tq[0] = T_q;
  map.Tt[0] = T_tail;
  set_row_units(map, 0, mma ? mma_tail_chunk(cfg->bits_k, cfg->bits_v) : 0);
  const long long U = P * units_of_row(map, 0);
  float* part_o = reinterpret_cast<float*>(ds.scratch);
  const size_t ml_off = round256(static_cast<size_t>(max_slots) * slot_o);
  float2* part_ml = reinterpret_cast<float2*>(ds.scratch + ml_off);
  int* err = reinterpret_cast<int*>(ds.scratch + round256(ml_off + max_slots * slot_ml));
  // The array keeps the previous call's contents: the error word must start
  // at zero; every partial slot the merge reads is written by this call.
  if (cudaMemsetAsync(err, 0, sizeof(int), st) != cudaSuccess) return KVQ_ERR_CUDA;
  if (U == 0) {
    if (cudaMemsetAsync(out, 0, static_cast<size_t>(P) * R * D * sizeof(float), st) != cudaSuccess)
      return KVQ_ERR_CUDA;
  } else {
    long long W = static_cast<long long>(ds.sm_count) * warps_per_sm;
    if (W > kMaxWarps) W = kMaxWarps;
    if (W > max_slots - P) W = max_slots - P;
    W = finish_map(map, static_cast<int>(P), 0, W);

    DecodeParams p;
    p.g.blocks = static_cast<uint8_t*>(const_cast<void*>(blocks));
    p.g.block_bytes = static_cast<uint64_t>(G) * D * (cfg->bits_k + cfg->bits_v) / 8 + 8ull * D;
    p.g.NB = NB;
    p.g.off_km = G * D * cfg->bits_k / 8;
    p.g.off_vc = p.g.off_km + 4 * D;
    p.g.off_vm = p.g.off_vc + G * D * cfg->bits_v / 8;
    p.g.D = D;
    p.g.G = G;
    p.g.bk = cfg->bits_k;
    p.g.bv = cfg->bits_v;
    p.g.frag_k = fragment_order(D, G, cfg->bits_k, cfg->axis_k, cfg->axis_v) ? 1 : 0;
    p.g.frag_v = fragment_order(D, G, cfg->bits_v, cfg->axis_k, cfg->axis_v) ? 1 : 0;
    p.g.ak = cfg->axis_k;
    p.g.av = cfg->axis_v;
    p.g.P = static_cast<int>(P);
    p.g.fp8 = cfg->fp8;
    p.g.TC = G;
    p.g.NSK = 0;
    p.g.nout = 0;
    p.g.off_ko = p.g.off_km + 4 * D;
    p.g.off_vo = p.g.off_vm + 4 * D;
    p.map = map;
    for (int i = 0; i < 2; ++i) {  // the caller's one tail, read only
      p.ktail[i] = static_cast<__half*>(const_cast<void*>(k_tail));
      p.vtail[i] = static_cast<__half*>(const_cast<void*>(v_tail));
    }
    p.act = 0;
    p.ksink = nullptr;
    p.vsink = nullptr;
    p.n_new = 0;
    p.knew = nullptr;
    p.vnew = nullptr;
    p.lg_G = G == 32 ? 5 : (G == 64 ? 6 : 7);
    p.lg_sub = p.lg_G - 5;
    p.n_warps = static_cast<int>(W);
    p.rope = 0;
    p.rope_tab = nullptr;
    p.rope_rows = 0;
    p.q = static_cast<const __half*>(q);
    p.qscale = softmax_scale * 1.4426950408889634f;
    p.part_o = part_o;
    p.part_ml = part_ml;
    p.err = err;
    p.wait_limit = kWaitLimit;
    p.fused = 0;
    p.tickets = nullptr;
    p.out = nullptr;
    if (ops.launch(p, st) != cudaSuccess) return KVQ_ERR_CUDA;
    MergeParams mp;
    mp.part_o = part_o;
    mp.part_ml = part_ml;
    mp.out = static_cast<float*>(out);
    mp.map = map;
    mp.R = R;
    mp.D = D;
    if (launch_merge(mp, static_cast<int>(P), st) != cudaSuccess) return KVQ_ERR_CUDA;
    count_launches(2);
  }
  if (device_error != nullptr &&
      cudaMemcpyAsync(device_error, err, sizeof(int), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return KVQ_ERR_CUDA;
  return KVQ_OK;
}
