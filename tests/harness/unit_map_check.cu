// Host-only check of the decode unit map (kvq_device.cuh): built by the CPU
// test suite with nvcc and run without a GPU.  For random uniform and ragged
// maps it verifies that pairs own disjoint, contiguous unit ranges covering
// [0, U), that pair_of_unit inverts first_unit, and that the partial slots
// (warp + pair) of all (warp, pair) pieces are distinct.
#include <cstdio>
#include <cstdlib>
#include <set>
#include <utility>
#include <vector>

#include "kvq_device.cuh"

using namespace kvq;

static unsigned rng_state = 12345u;
static int rnd(int n) {
  rng_state = rng_state * 1664525u + 1013904223u;
  return static_cast<int>((rng_state >> 8) % static_cast<unsigned>(n));
}

static int check(const UnitMap& m, int P, long long W, int* failures) {
  long long U = 0;
  for (int p = 0; p < P; ++p) U += units_of_row(m, row_of(m, p));
  long long next = 0;
  for (int p = 0; p < P; ++p) {
    const long long u0 = first_unit(m, p);
    const int upp = units_of_row(m, row_of(m, p));
    if (u0 != next) { ++*failures; return 0; }
    for (int j = 0; j < upp; ++j)
      if (pair_of_unit(m, u0 + j) != p) { ++*failures; return 0; }
    next = u0 + upp;
  }
  if (next != U) { ++*failures; return 0; }
  if (W > U) W = U;
  std::set<long long> slots;
  for (int p = 0; p < P; ++p) {
    const long long u0 = first_unit(m, p);
    const int upp = units_of_row(m, row_of(m, p));
    const long long w0 = owner_warp(u0, U, W), w1 = owner_warp(u0 + upp - 1, U, W);
    for (long long w = w0; w <= w1; ++w) {
      // warp w's range [w*U/W, (w+1)*U/W) must meet the pair's units
      const long long a = w * U / W, b = (w + 1) * U / W;
      if (b <= u0 || a >= u0 + upp) { ++*failures; return 0; }
      if (!slots.insert(w + p).second) { ++*failures; return 0; }
    }
  }
  return 1;
}

int main() {
  int failures = 0, cases = 0;
  for (int it = 0; it < 400; ++it) {
    UnitMap m = {};
    const int hkv = 1 + rnd(8);
    const int B = 1 + rnd(kMaxRows);
    const int tch = rnd(2) ? 6 + rnd(14) : 0;
    m.ragged = rnd(2);
    m.hkv = hkv;
    const int rows = m.ragged ? B : 1;
    for (int b = 0; b < rows; ++b) {
      m.Ts[b] = rnd(3) == 0 ? rnd(9) : 0;
      m.Tq[b] = 32 * rnd(200);
      m.Tt[b] = rnd(64);
      if (m.Ts[b] + m.Tq[b] + m.Tt[b] == 0) m.Tt[b] = 1;
      set_row_units(m, b, tch);
    }
    if (m.ragged) {
      m.uoff[0] = 0;
      for (int b = 0; b < B; ++b) m.uoff[b + 1] = m.uoff[b] + hkv * m.upp[b];
    }
    const long long W = 1 + rnd(4096);
    cases += check(m, B * hkv, W, &failures);
  }
  std::printf("cases %d failures %d\n", cases, failures);
  return failures == 0 ? 0 : 1;
}
