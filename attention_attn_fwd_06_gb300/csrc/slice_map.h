// slice_map.h -- how the persistent decode grid divides the cost space of all rows among its CTAs.
//
// Host and device code: the decode kernel uses it to find its own slice and, for a row split between CTAs, which
// CTAs hold its pieces; host tests check the tiling on the CPU.
#pragma once

#ifndef ATTN_DECODE_RANK_W0
#define ATTN_DECODE_RANK_W0 10
#endif

namespace attn {

// Slices are weighted by the CTA's launch rank on its SM.  The persistent grid is `ranks` CTAs per SM launched in
// rank-major order (CTA c has rank c / n, n = CTAs per rank), and per-CTA traces of the 8 x 4096 GQA workload show
// the CTAs sharing an SM streaming at about 1.0 : 0.9 : 0.8 of each other's rate by rank, so equal slices finish
// ~3.5 us apart.  Rank r takes weight W0 - r (10 : 9 : 8 by default).
struct SliceMap {
  long long Wc;     // cost positions to split
  long long g;      // slices
  long long n;      // slices per rank (0: equal slices)
  int ranks;
  long long total;  // sum of the weights of all slices
  __host__ __device__ long long weight(int r) const { return ATTN_DECODE_RANK_W0 - r; }
  // weights of the slices before slice c
  __host__ __device__ long long cum(long long c) const {
    if (n == 0) return c;
    const long long r = c / n;
    long long s = 0;
    for (int q = 0; q < r; ++q) s += n * weight(q);
    return s + (c - r * n) * weight((int)r);
  }
  // first cost position of slice c (c >= g: Wc); exact integer arithmetic, non-decreasing in c
  __host__ __device__ long long start(long long c) const { return c >= g ? Wc : (Wc * cum(c)) / total; }
  // the slice holding cost position pos (0 <= pos < Wc): the largest c with start(c) <= pos
  __host__ __device__ long long of(long long pos) const {
    const long long y = (pos * total) / Wc;  // the weight units before pos
    long long c;
    if (n == 0) {
      c = y;
    } else {
      long long s = 0;
      int r = 0;
      while (r + 1 < ranks && s + n * weight(r) <= y) s += n * weight(r++);
      c = r * n + (y - s) / weight(r);
    }
    c = c < 0 ? 0 : (c >= g ? g - 1 : c);
    while (c > 0 && start(c) > pos) --c;
    while (c + 1 < g && start(c + 1) <= pos) ++c;
    return c;
  }
};

// The map of g slices over Wc positions for a grid of `grid` CTAs launched `ranks` per SM: rank weights only for
// the full persistent grid with enough positions per slice; otherwise equal slices.
__host__ __device__ inline SliceMap make_slice_map(long long Wc, long long g, int ranks, long long grid) {
  SliceMap m;
  m.Wc = Wc;
  m.g = g;
  m.ranks = ranks;
  m.n = (ranks > 1 && g == grid && g % ranks == 0 && Wc >= 64 * g) ? g / ranks : 0;
  m.total = m.cum(g);
  return m;
}

}  // namespace attn
