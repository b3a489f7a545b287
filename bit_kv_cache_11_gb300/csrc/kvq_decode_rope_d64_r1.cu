// Tensor-core decode kernel for head_dim 64, 1 query head per kv head, keys
// stored before RoPE (rotated after dequantization), every (bits_k, bits_v)
// pair.  Its own translation unit so the library compiles in parallel.
#include "kvq_decode_mma.cuh"

namespace kvq {
DecodeOps decode_mma_rope_ops_d64_r1(int bk, int bv) { return decode_mma_ops_for<64, 1, true>(bk, bv, false); }
}  // namespace kvq
