// kernels.h -- internal launch interface between the C-ABI host code and the kernels.
// Not part of the public ABI (that is include/attn.h).
#pragma once

#include <cuda_runtime.h>

namespace attn {

// Split-KV decode (the split pass writes fp32 partials, the combine merges them).
struct DecodeLaunch {
  const void* q;        // bf16 [B, Hq, D]
  const void* kcache;   // bf16 [B, Hkv, Lmax, D]
  const void* vcache;   // bf16 [B, Hkv, Lmax, D]
  const int* kv_lens;   // int32 [B] (device)
  void* out;            // [B, Hq, D], bf16 or fp32
  float* lse;           // fp32 [B, Hq] or null
  float* part_o;        // fp32 [B, Hq, nsplit, D]
  float* part_ml;       // fp32 [B, Hq, nsplit, 2]  (m in log2 units, l)
  int B, Hq, Hkv, Lmax, D;
  int chunk;            // keys per split (multiple of the stage size)
  int nsplit;           // ceil(Lmax / chunk)
  float scale;
  int out_f32;
  unsigned* status;     // device status word
  cudaStream_t stream;
};

// Keys per pipeline stage of the split pass (chunk must be a multiple of it).
int decode_stage_keys(int D);
// Number of query heads one split CTA serves (the largest of 8, 4, 2, 1 dividing Hq / Hkv).
int decode_heads_per_cta(int group);
cudaError_t launch_decode(const DecodeLaunch& p);

// Prefill (tcgen05 tensor-core path).
struct PrefillLaunch {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* lse;
  int B, Hq, Hkv, Lq, Lkv, D;
  float scale;
  int causal;
  int out_f32;
  const int* cu_q;  // null for the dense layout
  const int* cu_k;
  int total_q, total_k;
  unsigned* status;
  cudaStream_t stream;
};

cudaError_t launch_prefill(const PrefillLaunch& p);

}  // namespace attn
