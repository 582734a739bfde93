// slice_map.h -- how the persistent decode grid divides the cost space of all rows among its CTAs.
//
// Host and device code: the decode kernel uses it to find its own slice and, for a row split between CTAs, which
// CTAs hold its pieces; host tests check the tiling on the CPU.
#pragma once

#include "intdiv.h"

#ifndef ATTN_DECODE_RANK_W0
#define ATTN_DECODE_RANK_W0 10
#endif

namespace attn {

// Slices are weighted by the CTA's launch rank on its SM.  The persistent grid is `ranks` CTAs per SM launched in
// rank-major order (CTA c has rank c / n, n = CTAs per rank), and per-CTA traces of the 8 x 4096 GQA workload show
// the CTAs sharing an SM streaming at about 1.0 : 0.9 : 0.8 of each other's rate by rank, so equal slices finish
// ~3.5 us apart.  Rank r takes weight W0 - r (10 : 9 : 8 by default).
struct SliceMap {
  long long Wc;          // cost positions to split
  int g;                 // slices
  int n;                 // slices per rank (0: equal slices)
  int ranks;
  long long total;       // sum of the weights of all slices
  float units_per_pos;   // total / Wc, for of()'s estimate
  __host__ __device__ long long weight(int r) const { return ATTN_DECODE_RANK_W0 - r; }
  // weights of the slices before slice c
  __host__ __device__ long long cum(int c) const {
    if (n == 0) return c;
    int r = 0;  // the rank of slice c, by comparison rather than c / n
    long long s = 0;
    while (r + 1 < ranks && c >= (r + 1) * n) s += (long long)n * weight(r++);
    return s + (long long)(c - r * n) * weight(r);
  }
  // first cost position of slice c (c >= g: Wc): floor(Wc * cum(c) / total), exact, non-decreasing in c
  __host__ __device__ long long start(long long c) const {
    return c >= g ? Wc : floor_div(Wc * cum((int)c), total);
  }
  // start(c) <= pos, without the division: floor(x / total) <= pos  <=>  x < (pos + 1) * total
  __host__ __device__ bool starts_by(long long c, long long pos) const {
    return c >= g ? Wc <= pos : Wc * cum((int)c) < (pos + 1) * total;
  }
  // the slice holding cost position pos (0 <= pos < Wc): the largest c with start(c) <= pos.  An fp32 estimate
  // of the weight units before pos (within one of the exact count) picks the slice; exact comparisons settle it.
  // (The decode kernel finds the same slices with a warp-wide search over starts_by, which needs no division or
  // conversion.)
  __host__ __device__ long long of(long long pos) const {
    const float yf = to_f32(pos) * units_per_pos;  // below total (< 2^31): a 32-bit conversion
    long long y = yf < 0.f ? 0 : (int)yf;
    y = y >= total ? total - 1 : y;
    int c;
    if (n == 0) {
      c = (int)y;
    } else {
      long long s = 0;
      int r = 0;
      while (r + 1 < ranks && s + (long long)n * weight(r) <= y) s += (long long)n * weight(r++);
      c = r * n + (int)(y - s) / (int)weight(r);
    }
    c = c < 0 ? 0 : (c >= g ? g - 1 : c);
    while (c > 0 && !starts_by(c, pos)) --c;
    while (c + 1 < g && starts_by(c + 1, pos)) ++c;
    return c;
  }
};

// The map of g slices over Wc positions for a grid of `grid` CTAs launched `ranks` per SM: rank weights only for
// the full persistent grid with enough positions per slice; otherwise equal slices.
__host__ __device__ inline SliceMap make_slice_map(long long Wc, long long g, int ranks, long long grid) {
  SliceMap m;
  m.Wc = Wc;
  m.g = (int)g;
  m.ranks = ranks;
  m.n = (ranks > 1 && g == grid && g % ranks == 0 && Wc >= 64 * g) ? (int)(g / ranks) : 0;
  m.total = m.cum((int)g);
  m.units_per_pos = (float)m.total / to_f32(Wc > 0 ? Wc : 1);
  return m;
}

}  // namespace attn
