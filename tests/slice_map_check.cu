// Host check of the decode grid's slice map (csrc/slice_map.h): floor_div equals integer division over the
// magnitudes the map uses; for many sizes, the slices tile the cost space in order with none empty, of() inverts
// start() exactly, and starts_by(c, pos) equals start(c) <= pos.  Prints "ok" and returns 0, or the first failure.
#include <cstdio>
#include <cstdlib>
#include <random>

#include "../attention_attn_fwd_06_gb300/csrc/slice_map.h"

static int fail(const char* what, long long Wc, long long g, long long x) {
  std::printf("FAIL %s Wc=%lld g=%lld at %lld\n", what, Wc, g, x);
  return 1;
}

static int check(long long Wc, long long g, int ranks, long long grid, bool expect_weighted, std::mt19937_64& rng) {
  const attn::SliceMap m = attn::make_slice_map(Wc, g, ranks, grid);
  if ((m.n != 0) != expect_weighted) return fail("weighting", Wc, g, m.n);
  if (m.start(0) != 0 || m.start(g) != Wc) return fail("ends", Wc, g, 0);
  for (long long c = 0; c < g; ++c) {
    const long long a = m.start(c), b = m.start(c + 1);
    if (b <= a && Wc >= g) return fail("empty or decreasing slice", Wc, g, c);
    if (b < a) return fail("decreasing", Wc, g, c);
    if (a < b && (m.of(a) != c || m.of(b - 1) != c)) return fail("of() at the slice edges", Wc, g, c);
  }
  std::uniform_int_distribution<long long> pos(0, Wc - 1);
  for (int i = 0; i < 2000; ++i) {
    const long long x = pos(rng);
    const long long c = m.of(x);
    if (!(m.start(c) <= x && x < m.start(c + 1))) return fail("of()", Wc, g, x);
    // starts_by (the division-free test the kernel's holder search uses) agrees with start() around c
    for (long long d = -2; d <= 2; ++d) {
      const long long cc = c + d;
      if (cc < 0 || cc > g) continue;
      for (long long px = x - 1; px <= x + 1; ++px)
        if (m.starts_by(cc, px) != (m.start(cc) <= px)) return fail("starts_by", Wc, g, px);
    }
  }
  if (m.n != 0) {  // the first rank's slices carry more than the last rank's
    const long long first = m.start(1) - m.start(0), last = m.start(g) - m.start(g - 1);
    if (first <= last) return fail("rank weights", Wc, g, first - last);
  }
  return 0;
}

static int check_floor_div(std::mt19937_64& rng) {
  for (int i = 0; i < 2000000; ++i) {
    const int abits = 1 + (int)(rng() % 63), bbits = 1 + (int)(rng() % 40);
    const long long a = (long long)(rng() >> (64 - abits));
    long long b = (long long)(rng() >> (64 - bbits));
    if (b == 0) b = 1;
    const long long want = a / b;
    // near-exact multiples are where an estimate is most often off by one
    const long long a2 = (want > 0 && want < (1LL << 62) / b) ? want * b - (long long)(rng() % 3) + 1 : a;
    if (attn::floor_div(a, b) != want) return fail("floor_div", a, b, want);
    if (a2 >= 0 && attn::floor_div(a2, b) != a2 / b)
      return fail("floor_div near a multiple", a2, b, a2 / b);
  }
  return 0;
}

int main() {
  std::mt19937_64 rng(7);
  if (check_floor_div(rng)) return 1;
  const long long grids[] = {456, 304, 444, 152};
  int bad = 0;
  for (long long grid : grids) {
    const int ranks = grid % 3 == 0 ? 3 : 2;
    // full persistent grid, enough positions: rank-weighted
    const long long big[] = {216000, 2700000, 64 * grid, (1LL << 40) + 12345, 29184LL * 7};
    for (long long Wc : big) bad |= check(Wc, grid, ranks, grid, Wc >= 64 * grid, rng);
    // fewer positions than 64 per slice, or fewer slices than the grid: equal slices
    bad |= check(64 * grid - 1, grid, ranks, grid, false, rng);
    bad |= check(5000, grid, ranks, grid, false, rng);
    bad |= check(12352, 64, ranks, grid, false, rng);
    bad |= check(1000000, grid - ranks, ranks, grid, false, rng);
    bad |= check(7, 7, ranks, grid, false, rng);
  }
  std::uniform_int_distribution<long long> wc(1000, 1LL << 36);
  for (int i = 0; i < 200; ++i) {
    const long long Wc = wc(rng);
    bad |= check(Wc, 456, 3, 456, Wc >= 64 * 456, rng);
  }
  if (bad) return 1;
  std::printf("ok\n");
  return 0;
}
