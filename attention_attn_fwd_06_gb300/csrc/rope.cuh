// rope.cuh -- rotary position embedding of one bf16 row held in a 128-byte
// swizzled shared-memory tile (the layout TMA writes and the tcgen05 MMAs
// read), in place.
//
// The rotation is the standard rotary embedding (the pages name RoPE as fusable
// into the attention kernel -- "Что такое kernel fusion и как он применяется в
// LLM serving?" §3.5, "GPU 学习日报 Day 24：Operator Fusion" exercise 1 -- without
// a formula): pair i of a row at position p, (a, b), becomes
// (a cos - b sin, b cos + a sin) with cos, sin read from row p of the caller's
// fp32 tables [max_pos, D/2]; pairs are dims (i, i + D/2) (style 1) or
// (2i, 2i + 1) (style 2).  Values are rotated in fp32 and rounded back to bf16
// (nearest, ties to even): the dtype of the tensor the unfused RoPE op would
// hand to attention, and the operand type of the tensor-core MMAs.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

#include "common.cuh"

namespace attn {

// Address of the 16-byte chunk holding columns x .. x+7 (x a multiple of 8) of `row` in a tile made of
// 64-column blocks of `block_bytes` each, 128 bytes per row, 16-byte chunks XOR-swizzled by row % 8.
__device__ __forceinline__ uint4* sw128_chunk(uint8_t* tile, int block_bytes, int row, int x) {
  const int db = x >> 6;
  const int c = (x & 63) >> 3;
  return reinterpret_cast<uint4*>(tile + db * block_bytes + row * 128 + ((c ^ (row & 7)) << 4));
}

__device__ __forceinline__ void unpack8(const uint4& w, float (&f)[8]) {
  bf16x2_to_f32(w.x, f[0], f[1]);
  bf16x2_to_f32(w.y, f[2], f[3]);
  bf16x2_to_f32(w.z, f[4], f[5]);
  bf16x2_to_f32(w.w, f[6], f[7]);
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack2_bf16(f[0], f[1]), pack2_bf16(f[2], f[3]), pack2_bf16(f[4], f[5]), pack2_bf16(f[6], f[7]));
}

// Rotates row `row` of a D-column swizzled tile to the position whose table rows are cos_row / sin_row
// (global memory, 16-byte aligned, D/2 floats each).  All of the row's table values are loaded before the
// tile is touched, so one row costs one memory latency rather than one per chunk.
template <int D>
__device__ __forceinline__ void rope_rotate_row_sw128(uint8_t* tile, int block_bytes, int row,
                                                      const float* __restrict__ cos_row,
                                                      const float* __restrict__ sin_row, int style) {
  constexpr int NP = D / 2;  // pairs
  float4 c4[NP / 4], s4[NP / 4];
#pragma unroll
  for (int i = 0; i < NP / 4; ++i) {
    c4[i] = __ldg(reinterpret_cast<const float4*>(cos_row) + i);
    s4[i] = __ldg(reinterpret_cast<const float4*>(sin_row) + i);
  }
  auto cf = [&](int i) -> float { return reinterpret_cast<const float*>(c4)[i]; };
  auto sf = [&](int i) -> float { return reinterpret_cast<const float*>(s4)[i]; };
  if (style == 1) {
    // pairs (i, i + D/2): chunk x0 of the first half with the chunk D/2 columns later
#pragma unroll
    for (int x0 = 0; x0 < NP; x0 += 8) {
      uint4* pa = sw128_chunk(tile, block_bytes, row, x0);
      uint4* pb = sw128_chunk(tile, block_bytes, row, x0 + NP);
      float a[8], b[8], ra[8], rb[8];
      unpack8(*pa, a);
      unpack8(*pb, b);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        ra[j] = fmaf(a[j], cf(x0 + j), -b[j] * sf(x0 + j));
        rb[j] = fmaf(b[j], cf(x0 + j), a[j] * sf(x0 + j));
      }
      *pa = pack8(ra);
      *pb = pack8(rb);
    }
  } else {
    // pairs (2i, 2i + 1): every chunk holds four whole pairs
#pragma unroll
    for (int x0 = 0; x0 < D; x0 += 8) {
      uint4* pc = sw128_chunk(tile, block_bytes, row, x0);
      float v[8], r[8];
      unpack8(*pc, v);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = x0 / 2 + k;
        r[2 * k] = fmaf(v[2 * k], cf(i), -v[2 * k + 1] * sf(i));
        r[2 * k + 1] = fmaf(v[2 * k + 1], cf(i), v[2 * k] * sf(i));
      }
      *pc = pack8(r);
    }
  }
}

}  // namespace attn
