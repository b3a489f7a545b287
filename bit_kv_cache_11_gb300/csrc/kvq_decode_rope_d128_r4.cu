// Tensor-core decode kernel for head_dim 128, 4 query heads per kv head, keys
// stored before RoPE (rotated after dequantization), every (bits_k, bits_v)
// pair.  Its own translation unit so the library compiles in parallel.
#include "kvq_decode_mma.cuh"

namespace kvq {
DecodeOps decode_mma_rope_ops_d128_r4(int bk, int bv) { return decode_mma_ops_for<128, 4, true>(bk, bv, false); }
}  // namespace kvq
