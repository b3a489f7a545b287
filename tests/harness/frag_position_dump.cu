// Host-only dump of the device code-order function (kvq_device.cuh): for each
// bit width and head dim, the word and bit of every element of a block's K
// tile (32 tokens x D channels) and V tile (D channels x 32 tokens).  Lines:
//   side bits D token channel word bit
#include <cstdio>

#include "kvq_device.cuh"

int main() {
  const int bits_list[3] = {2, 4, 8};
  const int d_list[2] = {64, 128};
  for (int bits : bits_list)
    for (int D : d_list)
      for (int j = 0; j < 32; ++j)
        for (int d = 0; d < D; ++d) {
          int w, b;
          kvq::frag_position(j, d, D, bits, &w, &b);   // K: row token, col channel
          std::printf("K %d %d %d %d %d %d\n", bits, D, j, d, w, b);
          kvq::frag_position(d, j, 32, bits, &w, &b);  // V: row channel, col token
          std::printf("V %d %d %d %d %d %d\n", bits, D, j, d, w, b);
        }
  return 0;
}
