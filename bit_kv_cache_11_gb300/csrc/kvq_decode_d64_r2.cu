// Decode kernels for head_dim 64, 2 query heads per kv head: the general CUDA-core
// kernel for every (bits_k, bits_v) pair and the tensor-core kernel for the
// pages' geometry (keys stored after RoPE; the rotated-key variant is in
// kvq_decode_rope_d64_r2.cu).  One translation unit per (D, R) so the
// library compiles in parallel.
#include "kvq_decode.cuh"
#include "kvq_decode_mma.cuh"

namespace kvq {
DecodeOps decode_ops_d64_r2(int bk, int bv) { return decode_ops_for<64, 2>(bk, bv); }
DecodeOps decode_mma_ops_d64_r2(int bk, int bv, bool out) { return decode_mma_ops_for<64, 2, false>(bk, bv, out); }
}  // namespace kvq
