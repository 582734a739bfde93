// intdiv.h -- 64-bit integer helpers for the decode kernels' work split, built from 32-bit operations.
//
// The producer warp of a persistent decode CTA computes its slice and the merge bookkeeping of each row piece
// before that piece's first stage can complete.  A 64-bit integer division, or a conversion between a 64-bit
// integer and a float, takes on the order of a microsecond of that warp's time there (per-CTA timer traces of the
// 8 x 4096 GQA decode), while 32-bit divisions and conversions are cheap, so these helpers use only those.
// Host and device run the same code.
#pragma once

namespace attn {

// floor(a / b) for a >= 0 and b >= 1, exact.  Operands that fit 32 bits take one 32-bit division; a wider
// dividend over a divisor below 2^16 is divided in 32-, 16- and 16-bit digits (each step's partial remainder
// times 2^16 plus the next digit stays below 2^32); anything else falls back to the 64-bit division.
__host__ __device__ inline long long floor_div(long long a, long long b) {
  const unsigned long long ua = (unsigned long long)a;
  if ((ua >> 32) == 0 && b <= 0xffffffffLL) return (long long)((unsigned)ua / (unsigned)b);
  if (b < 65536) {
    const unsigned d = (unsigned)b;
    const unsigned hi = (unsigned)(ua >> 32);
    const unsigned q0 = hi / d, r0 = hi - q0 * d;
    const unsigned t1 = (r0 << 16) | (unsigned)((ua >> 16) & 0xffffu);
    const unsigned q1 = t1 / d, r1 = t1 - q1 * d;
    const unsigned t2 = (r1 << 16) | (unsigned)(ua & 0xffffu);
    const unsigned q2 = t2 / d;
    return (long long)(((unsigned long long)q0 << 32) | ((unsigned long long)q1 << 16) | q2);
  }
  return a / b;
}

// x >= 0 as a float (relative error below 2^-22), from its two 32-bit halves.
__host__ __device__ inline float to_f32(long long x) {
  const unsigned long long u = (unsigned long long)x;
  return (float)(unsigned)(u >> 32) * 4294967296.0f + (float)(unsigned)(u & 0xffffffffu);
}

}  // namespace attn
