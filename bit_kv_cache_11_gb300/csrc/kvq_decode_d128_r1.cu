// Decode kernels for head_dim 128, 1 query head(s) per kv head, all
// (bits_k, bits_v) pairs.  One translation unit per (D, R) so the library
// compiles in parallel.
#include "kvq_decode.cuh"

namespace kvq {
DecodeOps decode_ops_d128_r1(int bk, int bv) { return decode_ops_for<128, 1>(bk, bv); }
}  // namespace kvq
