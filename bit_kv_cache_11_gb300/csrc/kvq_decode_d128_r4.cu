// Decode kernels for head_dim 128, 4 query head(s) per kv head: the
// general CUDA-core kernel for every (bits_k, bits_v) pair and the tensor-core
// kernel for the pages' geometry (with a rotated-key variant for keys stored
// before RoPE where instantiated).  One translation unit per (D, R) so the
// library compiles in parallel.
#include "kvq_decode.cuh"
#include "kvq_decode_mma.cuh"

namespace kvq {
DecodeOps decode_ops_d128_r4(int bk, int bv) { return decode_ops_for<128, 4>(bk, bv); }
DecodeOps decode_mma_ops_d128_r4(int bk, int bv, bool rope) {
  return rope ? decode_mma_ops_for<128, 4, true>(bk, bv) : decode_mma_ops_for<128, 4, false>(bk, bv);
}
}  // namespace kvq
