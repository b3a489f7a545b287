// Host-only check of the decode unit map (kvq_device.cuh): built by the CPU
// test suite with nvcc and run without a GPU.  For random uniform and ragged
// maps and 0 to 3 virtual units per pair it verifies that pairs own
// disjoint, contiguous unit ranges covering [0, U), that pair_of_unit
// inverts first_unit, that the cost of a unit maps back to it, that the warp
// ranges of the cost split tile [0, U) in order, that pair_warps names the
// warps holding a pair's units, and that the partial slots (warp + pair) of
// all (warp, pair) pieces are distinct.
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

static int check(UnitMap m, int P, long long Wmax, int vcost, int* failures) {
  const int W = finish_map(m, P, vcost, Wmax);
  long long next = 0;
  for (int p = 0; p < P; ++p) {
    const long long u0 = first_unit(m, p);
    const int upp = units_of_row(m, row_of(m, p));
    if (u0 != next) { ++*failures; return 0; }
    for (int j = 0; j < upp; ++j)
      if (pair_of_unit(m, u0 + j) != p) { ++*failures; return 0; }
    // costs: the pair's units take costs [first_cost, first_cost + upp), then vcost virtual ones
    const int want_c0 =
        p == 0 ? 0 : first_cost(m, p - 1) + units_of_row(m, row_of(m, p - 1)) + vcost;
    if (first_cost(m, p) != want_c0) { ++*failures; return 0; }
    for (int j = 0; j <= upp + vcost; ++j) {
      const int want = j < upp ? static_cast<int>(u0) + j : static_cast<int>(u0) + upp;
      if (unit_at_cost(m, first_cost(m, p) + j) != want) { ++*failures; return 0; }
    }
    next = u0 + upp;
  }
  if (next != m.U || static_cast<long long>(m.C) != m.U + static_cast<long long>(P) * vcost) {
    ++*failures;
    return 0;
  }
  // warp ranges: contiguous, in order, covering [0, U)
  int prev_end = 0;
  std::vector<int> owner(m.U, -1);
  for (int w = 0; w < W; ++w) {
    int a, b;
    warp_units(m, w, &a, &b);
    if (a != prev_end || b < a) { ++*failures; return 0; }
    for (int u = a; u < b; ++u) owner[u] = w;
    prev_end = b;
  }
  if (prev_end != m.U) { ++*failures; return 0; }
  // pair_warps names exactly the warps that hold units of the pair, and the
  // partial slots (warp + pair) are distinct
  std::set<long long> slots;
  for (int p = 0; p < P; ++p) {
    const long long u0 = first_unit(m, p);
    const int upp = units_of_row(m, row_of(m, p));
    int w0, w1;
    pair_warps(m, p, &w0, &w1);
    std::set<int> holders;
    for (int j = 0; j < upp; ++j) holders.insert(owner[u0 + j]);
    if (upp > 0) {
      if (*holders.begin() != w0 || *holders.rbegin() != w1 ||
          static_cast<int>(holders.size()) != w1 - w0 + 1) {
        ++*failures;
        return 0;
      }
    }
    for (int w = w0; w <= w1; ++w)
      if (!slots.insert(static_cast<long long>(w) + p).second) { ++*failures; return 0; }
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
    m.rows = rows;
    const long long W = 1 + rnd(4096);
    cases += check(m, B * hkv, W, rnd(4), &failures);
  }
  std::printf("cases %d failures %d\n", cases, failures);
  return failures == 0 ? 0 : 1;
}
