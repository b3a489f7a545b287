// Decode kernels for head_dim 128, 2 query head(s) per kv head, all
// (bits_k, bits_v) pairs.  One translation unit per (D, R) so the library
// compiles in parallel.
#include "kvq_decode.cuh"

namespace kvq {
DecodeOps decode_ops_d128_r2(int bk, int bv) { return decode_ops_for<128, 2>(bk, bv); }
}  // namespace kvq
