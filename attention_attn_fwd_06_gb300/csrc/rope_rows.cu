// rope_rows.cu -- rotary position embedding of the keys and of the queries of
// a prefill call, one pass each per call, before the attention kernel reads
// them.
//
// The rotation is the one of rope.cuh (pair i of a row at position p, (a, b),
// becomes (a cos - b sin, b cos + a sin) with cos, sin from row p of the
// caller's fp32 tables; pairs (i, i + D/2) or (2i, 2i + 1); fp32 arithmetic,
// bf16 result).  Key j of a sequence sits at position j, query i at
// i + Lkv - Lq (the causal alignment).
//
// Why passes of their own: in a causal prefill every K tile of a head is read
// by every query-tile job of that head; rotating it where it lands in shared
// memory repeats the rotation (and the cos/sin reads, 2x the tile's bytes) for
// every visit and made the attention kernel L2-bound (measured 2.3x slower).
// A Q tile is loaded once per job, but rotating it where it lands put the
// rotation on the MMA warp's path at every job start (the causal 4k call took
// 570 us that way, 526 us with this pass).  Each pass reads its tensor and
// the tables once and writes the rotated rows -- the keys a serving engine
// wants anyway for its KV cache -- and the attention kernel then streams them
// like unrotated ones.
//
// Layout: dense [B, H, L, D] (row r of head (b, h) at position r + pos_off),
// or packed [total, H, D] with cu_seqlens (token t of sequence s at position
// t - cu[s], plus that sequence's Lkv - Lq for queries).  Each thread rotates
// eight pairs of one row with 16-byte loads and stores; a warp covers whole
// rows, so global accesses are coalesced.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace {

__device__ __forceinline__ void unpack8f(const uint4& w, float (&f)[8]) {
  bf16x2_to_f32(w.x, f[0], f[1]);
  bf16x2_to_f32(w.y, f[2], f[3]);
  bf16x2_to_f32(w.z, f[4], f[5]);
  bf16x2_to_f32(w.w, f[6], f[7]);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ uint4 pack8f(const float (&f)[8]) {
  return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
}

// One thread = one group of eight pairs of one row: TPR threads per row.
template <int D>
__global__ void __launch_bounds__(256) rope_rows_kernel(const RopeRowsLaunch p, long long nrows) {
  constexpr int NP = D / 2;
  constexpr int TPR = NP / 8;  // threads per row
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = tid / TPR;  // row in memory order
  const int grp = (int)(tid % TPR);
  if (row >= nrows) return;
  // position of the row within its sequence
  long long pos;
  if (p.cu == nullptr) {
    pos = row % p.L + p.pos_off;  // [B, H, L, D]
  } else {
    const long long tok = row / p.H;  // [total, H, D]
    int lo = 0, hi = p.B;             // the sequence s with cu[s] <= tok < cu[s + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (p.cu[mid] <= tok) lo = mid; else hi = mid;
    }
    pos = tok - p.cu[lo];
    if (p.cu_kv != nullptr) pos += (long long)(p.cu_kv[lo + 1] - p.cu_kv[lo]) - (p.cu[lo + 1] - p.cu[lo]);
  }
  if (pos < 0 || pos >= p.rope.max_pos) {
    record_status(p.status, ATTN_ERR_DEVICE_BOUNDS);
    pos = pos < 0 ? 0 : p.rope.max_pos - 1;
  }
  const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(p.src) + row * D;
  __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.dst) + row * D;
  const float* crow = p.rope.cos + pos * NP;
  const float* srow = p.rope.sin + pos * NP;
  if (p.rope.style == 1) {
    // pairs (i, i + D/2), i = 8 grp .. 8 grp + 7
    const int i0 = 8 * grp;
    float a[8], b[8], c[8], s[8], ra[8], rb[8];
    unpack8f(*reinterpret_cast<const uint4*>(src + i0), a);
    unpack8f(*reinterpret_cast<const uint4*>(src + i0 + NP), b);
    *reinterpret_cast<float4*>(c) = __ldg(reinterpret_cast<const float4*>(crow + i0));
    *reinterpret_cast<float4*>(c + 4) = __ldg(reinterpret_cast<const float4*>(crow + i0 + 4));
    *reinterpret_cast<float4*>(s) = __ldg(reinterpret_cast<const float4*>(srow + i0));
    *reinterpret_cast<float4*>(s + 4) = __ldg(reinterpret_cast<const float4*>(srow + i0 + 4));
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      ra[j] = fmaf(a[j], c[j], -b[j] * s[j]);
      rb[j] = fmaf(b[j], c[j], a[j] * s[j]);
    }
    *reinterpret_cast<uint4*>(dst + i0) = pack8f(ra);
    *reinterpret_cast<uint4*>(dst + i0 + NP) = pack8f(rb);
  } else {
    // pairs (2i, 2i + 1), i = 8 grp .. 8 grp + 7: dims 16 grp .. 16 grp + 15
    const int d0 = 16 * grp;
    float v[16], c[8], s[8], r[16];
    unpack8f(*reinterpret_cast<const uint4*>(src + d0), *reinterpret_cast<float(*)[8]>(v));
    unpack8f(*reinterpret_cast<const uint4*>(src + d0 + 8), *reinterpret_cast<float(*)[8]>(v + 8));
    *reinterpret_cast<float4*>(c) = __ldg(reinterpret_cast<const float4*>(crow + 8 * grp));
    *reinterpret_cast<float4*>(c + 4) = __ldg(reinterpret_cast<const float4*>(crow + 8 * grp + 4));
    *reinterpret_cast<float4*>(s) = __ldg(reinterpret_cast<const float4*>(srow + 8 * grp));
    *reinterpret_cast<float4*>(s + 4) = __ldg(reinterpret_cast<const float4*>(srow + 8 * grp + 4));
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      r[2 * k] = fmaf(v[2 * k], c[k], -v[2 * k + 1] * s[k]);
      r[2 * k + 1] = fmaf(v[2 * k + 1], c[k], v[2 * k] * s[k]);
    }
    *reinterpret_cast<uint4*>(dst + d0) = pack8f(*reinterpret_cast<float(*)[8]>(r));
    *reinterpret_cast<uint4*>(dst + d0 + 8) = pack8f(*reinterpret_cast<float(*)[8]>(r + 8));
  }
}

}  // namespace

cudaError_t launch_rope_rows(const RopeRowsLaunch& p) {
  const long long nrows = p.cu == nullptr ? (long long)p.B * p.H * p.L : (long long)p.total * p.H;
  if (nrows <= 0) return cudaSuccess;
  const int tpr = p.D / 16;
  const long long threads = nrows * tpr;
  const long long blocks = (threads + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (p.D == 64)
    rope_rows_kernel<64><<<(unsigned)blocks, 256, 0, p.stream>>>(p, nrows);
  else if (p.D == 128)
    rope_rows_kernel<128><<<(unsigned)blocks, 256, 0, p.stream>>>(p, nrows);
  else
    return cudaErrorNotSupported;
  return cudaGetLastError();
}

}  // namespace attn
