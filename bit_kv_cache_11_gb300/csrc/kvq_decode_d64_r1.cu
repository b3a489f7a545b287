// Decode kernels for head_dim 64, 1 query head(s) per kv head: the
// general CUDA-core kernel for every (bits_k, bits_v) pair and the tensor-core
// kernel for the pages' geometry (with a rotated-key variant for keys stored
// before RoPE where instantiated).  One translation unit per (D, R) so the
// library compiles in parallel.
#include "kvq_decode.cuh"
#include "kvq_decode_mma.cuh"

namespace kvq {
DecodeOps decode_ops_d64_r1(int bk, int bv) { return decode_ops_for<64, 1>(bk, bv); }
DecodeOps decode_mma_ops_d64_r1(int bk, int bv, bool rope) {
  return rope ? decode_mma_ops_for<64, 1, true>(bk, bv) : decode_mma_ops_for<64, 1, false>(bk, bv);
}
}  // namespace kvq
