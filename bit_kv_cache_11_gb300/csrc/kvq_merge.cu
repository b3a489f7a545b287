// kvq_merge.cu — combines the split-K partials of every pair, and the
// dispatch table of decode instantiations.
//
// Merging partial softmax states is the identity behind splitting a softmax
// sum: with m* = max_s m_s and w_s = 2^(m_s - m*) (scores in log2 units),
//   out = sum_s w_s o_s / sum_s w_s l_s.
#include "kvq_decode.cuh"
#include "kvq_decode_mma.cuh"

namespace kvq {

DecodeOps decode_ops_d64_r1(int, int);
DecodeOps decode_ops_d64_r2(int, int);
DecodeOps decode_ops_d64_r4(int, int);
DecodeOps decode_ops_d64_r8(int, int);
DecodeOps decode_ops_d128_r1(int, int);
DecodeOps decode_ops_d128_r2(int, int);
DecodeOps decode_ops_d128_r4(int, int);
DecodeOps decode_ops_d128_r8(int, int);

DecodeOps decode_mma_ops_d64_r1(int, int, bool);
DecodeOps decode_mma_ops_d64_r2(int, int, bool);
DecodeOps decode_mma_ops_d64_r4(int, int, bool);
DecodeOps decode_mma_ops_d64_r8(int, int, bool);
DecodeOps decode_mma_ops_d128_r1(int, int, bool);
DecodeOps decode_mma_ops_d128_r2(int, int, bool);
DecodeOps decode_mma_ops_d128_r4(int, int, bool);
DecodeOps decode_mma_ops_d128_r8(int, int, bool);
DecodeOps decode_mma_rope_ops_d64_r1(int, int);
DecodeOps decode_mma_rope_ops_d64_r2(int, int);
DecodeOps decode_mma_rope_ops_d64_r4(int, int);
DecodeOps decode_mma_rope_ops_d64_r8(int, int);
DecodeOps decode_mma_rope_ops_d128_r1(int, int);
DecodeOps decode_mma_rope_ops_d128_r2(int, int);
DecodeOps decode_mma_rope_ops_d128_r4(int, int);
DecodeOps decode_mma_rope_ops_d128_r8(int, int);

DecodeOps decode_mma_ops(int D, int R, int bk, int bv, bool rope, bool out) {
  if (D == 64) {
    if (R == 1) return rope ? decode_mma_rope_ops_d64_r1(bk, bv) : decode_mma_ops_d64_r1(bk, bv, out);
    if (R == 2) return rope ? decode_mma_rope_ops_d64_r2(bk, bv) : decode_mma_ops_d64_r2(bk, bv, out);
    if (R == 4) return rope ? decode_mma_rope_ops_d64_r4(bk, bv) : decode_mma_ops_d64_r4(bk, bv, out);
    if (R == 8) return rope ? decode_mma_rope_ops_d64_r8(bk, bv) : decode_mma_ops_d64_r8(bk, bv, out);
  } else if (D == 128) {
    if (R == 1) return rope ? decode_mma_rope_ops_d128_r1(bk, bv) : decode_mma_ops_d128_r1(bk, bv, out);
    if (R == 2) return rope ? decode_mma_rope_ops_d128_r2(bk, bv) : decode_mma_ops_d128_r2(bk, bv, out);
    if (R == 4) return rope ? decode_mma_rope_ops_d128_r4(bk, bv) : decode_mma_ops_d128_r4(bk, bv, out);
    if (R == 8) return rope ? decode_mma_rope_ops_d128_r8(bk, bv) : decode_mma_ops_d128_r8(bk, bv, out);
  }
  return DecodeOps{nullptr, nullptr};
}

DecodeOps decode_ops(int D, int R, int bk, int bv) {
  if (D == 64) {
    if (R == 1) return decode_ops_d64_r1(bk, bv);
    if (R == 2) return decode_ops_d64_r2(bk, bv);
    if (R == 4) return decode_ops_d64_r4(bk, bv);
    if (R == 8) return decode_ops_d64_r8(bk, bv);
  } else if (D == 128) {
    if (R == 1) return decode_ops_d128_r1(bk, bv);
    if (R == 2) return decode_ops_d128_r2(bk, bv);
    if (R == 4) return decode_ops_d128_r4(bk, bv);
    if (R == 8) return decode_ops_d128_r8(bk, bv);
  }
  return DecodeOps{nullptr, nullptr};
}

// grid = P pairs, block = D threads (one output channel each).
__global__ void merge_kernel(const MergeParams mp) {
  const long long pr = blockIdx.x;
  const int d = threadIdx.x;
  int w0, w1;
  pair_warps(mp.map, pr, &w0, &w1);
  for (int r = 0; r < mp.R; ++r) {
    float ms = -INFINITY;
    for (long long w = w0; w <= w1; ++w) ms = fmaxf(ms, mp.part_ml[(w + pr) * mp.R + r].x);
    // Partials that saw no token (m = -inf, l = 0) weigh 0; if all of them
    // are empty the output is 0.
    const float mb = ms == -INFINITY ? 0.f : ms;
    float L = 0.f, o = 0.f;
    for (long long w = w0; w <= w1; ++w) {
      const float2 ml = mp.part_ml[(w + pr) * mp.R + r];
      const float f = exp2f(ml.x - mb);
      L = fmaf(f, ml.y, L);
      o = fmaf(f, mp.part_o[((w + pr) * mp.R + r) * mp.D + d], o);
    }
    mp.out[(pr * mp.R + r) * mp.D + d] = L > 0.f ? o / L : 0.f;
  }
}

// Weighted sum over n rows (row k: {m, l} at ml[k mlstride], o at o0[k ostride]) of
// this thread's channel, with the weights exp2(m_k - max m): the {m, l} go
// through shared memory in one round of loads, the o values are loaded 16
// rows at a time before any is used.  Returns the sum; *ms, *L the maximum
// and the weighted l (-inf and 0 when every row is empty).
__device__ __forceinline__ float merge_column(int n, const float2* ml, long long mlstride,
                                              bool coherent, const float* o0, long long ostride,
                                              float2* sml, float* ms_out, float* L_out) {
  const int d = threadIdx.x;
  __syncthreads();  // sml free (a previous use)
  for (int k = d; k < n; k += blockDim.x)
    sml[k] = coherent ? __ldcg(ml + k * mlstride) : ml[k * mlstride];
  __syncthreads();
  float ms = -INFINITY;
  for (int k = 0; k < n; ++k) ms = fmaxf(ms, sml[k].x);
  const float mb = ms == -INFINITY ? 0.f : ms;  // every row empty: weights 0
  float L = 0.f, o = 0.f;
  for (int k0 = 0; k0 < n; k0 += 16) {
    float v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int k = min(k0 + u, n - 1);
      v[u] = coherent ? __ldcg(o0 + k * ostride) : o0[k * ostride];
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      if (k0 + u < n) {
        const float2 m = sml[k0 + u];
        const float f = exp2f(m.x - mb);
        L = fmaf(f, m.y, L);
        o = fmaf(f, v[u], o);
      }
    }
  }
  *ms_out = ms;
  *L_out = L;
  return o;
}

// grid = P * R * C2 blocks of D threads.
__global__ void merge2_kernel(const Merge2Params mp) {
  __shared__ float2 sml[kMerge2MaxRows];
  const int b = blockIdx.x;
  const int c = b % mp.C2;
  const int pq = b / mp.C2;
  const int r = pq % mp.R;
  const long long pr = pq / mp.R;
  const int d = threadIdx.x;
  // Launched as a programmatic dependent of the decode grid: its blocks may
  // become resident while that grid drains; wait for it (and its writes)
  // before reading, and let the next grid of the stream launch meanwhile.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  int w0, w1;
  pair_warps(mp.map, pr, &w0, &w1);
  const long long s0 = w0 + static_cast<long long>(mp.CS) * c;
  const long long s1 = s0 + mp.CS - 1 < w1 ? s0 + mp.CS - 1 : w1;
  // the chunk's partial slots s0 .. s1 (a chunk may hold only empty partials)
  float ms, L;
  const float o = merge_column(static_cast<int>(s1 - s0 + 1), mp.part_ml + (s0 + pr) * mp.R + r, mp.R,
                               false, mp.part_o + ((s0 + pr) * mp.R + r) * mp.D + d,
                               static_cast<long long>(mp.R) * mp.D, sml, &ms, &L);
  mp.lvl_o[static_cast<size_t>(b) * mp.D + d] = o;
  if (d == 0) mp.lvl_ml[b] = make_float2(ms, L);
  __threadfence();
  __syncthreads();
  __shared__ int last;
  if (d == 0) last = atomicAdd(&mp.tickets[pq], 1) == mp.C2 - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  const size_t base = static_cast<size_t>(pq) * mp.C2;
  const float o2 = merge_column(mp.C2, mp.lvl_ml + base, 1, true, mp.lvl_o + base * mp.D + d, mp.D,
                                sml, &ms, &L);
  mp.out[(pr * mp.R + r) * mp.D + d] = L > 0.f ? o2 / L : 0.f;
  if (d == 0) mp.tickets[pq] = 0;
}

cudaError_t launch_merge2(const Merge2Params& mp, int n_pairs, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_pairs * mp.R * mp.C2);
  cfg.blockDim = dim3(mp.D);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, merge2_kernel, mp);
}

cudaError_t launch_merge(const MergeParams& mp, int n_pairs, cudaStream_t stream) {
  merge_kernel<<<n_pairs, mp.D, 0, stream>>>(mp);
  return cudaGetLastError();
}

}  // namespace kvq
