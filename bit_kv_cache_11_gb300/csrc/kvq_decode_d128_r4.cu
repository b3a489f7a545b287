// Decode kernels for head_dim 128, 4 query head(s) per kv head, all
// (bits_k, bits_v) pairs.  One translation unit per (D, R) so the library
// compiles in parallel.
#include "kvq_decode.cuh"

namespace kvq {
DecodeOps decode_ops_d128_r4(int bk, int bv) { return decode_ops_for<128, 4>(bk, bv); }
}  // namespace kvq
