// kernels.h -- internal launch interface between the C-ABI host code and the kernels.
// Not part of the public ABI (that is include/attn.h).
#pragma once

#include <cuda_runtime.h>

namespace attn {

// Rotary position embedding tables (see attn_rope in include/attn.h); style 0 = off.
struct RopeArgs {
  const float* cos;  // fp32 [max_pos, D/2]
  const float* sin;
  int max_pos;
  int style;         // 1: pairs (i, i + D/2); 2: pairs (2i, 2i + 1)
};

// Split-KV decode (the split pass writes fp32 partials, the combine merges them).
struct DecodeLaunch {
  const void* q;        // bf16 [B, Hq, D]
  const void* kcache;   // bf16 [B, Hkv, Lmax, D], or the page pool [num_pages, Hkv, page_size, D]
  const void* vcache;   // same layout as kcache
  const int* block_table;  // null: contiguous cache; else int32 [B, max_pages] page ids (Lmax = max_pages*page_size)
  int page_size, max_pages, num_pages;
  const int* kv_lens;   // int32 [B] (device)
  void* out;            // [B, Hq, D], bf16 or fp32
  float* lse;           // fp32 [B, Hq] or null
  float* part_o;        // fp32 [2 * grid][GP][D]   partial O per (CTA slot, head of the group)
  float* part_ml;       // fp32 [2 * grid][GP][2]   (m in log2 units, l)
  unsigned* counters;   // [2 + row]: partials landed per (b, kv head, head group) row; zero between calls
  int B, Hq, Hkv, Lmax, D;
  int min_keys;         // smallest slice of the key space one CTA takes (>= 1)
  float scale;
  int out_f32;
  unsigned* status;     // device status word
  RopeArgs rope;        // rotates q (to kv_len - 1) when style != 0
  int fault_skip_arrive;  // test hook: CTA 0 withholds one slot release, so a bounded wait runs out
  cudaStream_t stream;
};

// Keys per pipeline stage of the split pass.
int decode_stage_keys(int D);
// CTAs of the persistent decode launch (three per SM, two with 8 heads per CTA); the partial slots
// number 2 * grid.
int decode_grid(int num_sms, int group);
// Number of query heads one decode CTA serves (the largest of 8, 4, 2, 1 dividing Hq / Hkv).
int decode_heads_per_cta(int group);
// Counter slots the decode kernel may use: 2 + B * Hkv * (Hq / Hkv / heads_per_cta) must fit.
constexpr int kDecodeCounterSlots = 65536;
// One persistent launch that also merges the split partials.
cudaError_t launch_decode(const DecodeLaunch& p, int num_sms);

// Multi-token decode (tcgen05 tensor-core path): Lq new tokens per sequence over a contiguous KV cache.
struct DecodeMultiLaunch {
  const void* q;        // bf16 [B, Hq, Lq, D]
  const void* kcache;   // bf16 [B, Hkv, Lmax, D]
  const void* vcache;   // same layout as kcache
  const int* kv_lens;   // int32 [B] (device); keys of every token, the new ones included
  void* out;            // [B, Hq, Lq, D], bf16 or fp32
  float* lse;           // fp32 [B, Hq, Lq] or null
  float* part_o;        // fp32 [2 * grid][R][D], R = (Hq / Hkv) * Lq
  float* part_ml;       // fp32 [2 * grid][R][2]
  unsigned* counters;   // [2 + b * Hkv + hk]; zero between calls (shared with the single-token decode)
  int B, Hq, Hkv, Lq, Lmax, D;
  float scale;
  int out_f32;
  int num_sms;
  unsigned* status;
  RopeArgs rope;        // rotates q (token t to kv_len - Lq + t) when style != 0
  int fault_skip_arrive;  // test hook: CTA 0 withholds one P-ready arrival (its MMA warp's wait runs out)
  cudaStream_t stream;
};

// CTAs of the persistent multi-token decode launch (one per SM); the partial slots number 2 * grid.
int decode_multi_grid(int num_sms);
cudaError_t launch_decode_multi(const DecodeMultiLaunch& p);

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
  int num_sms;      // persistent grid size
  unsigned* status;
  int fault_skip_arrive;  // test hook: CTA 0 withholds one P-ready arrival (its MMA warp's wait runs out)
  cudaStream_t stream;
};

cudaError_t launch_prefill(const PrefillLaunch& p);

// Rotary embedding of the keys or the queries of a prefill call into dst (same layout as src), once per call.
struct RopeRowsLaunch {
  const void* src;     // bf16 [B, H, L, D] (dense) or [total, H, D] (packed)
  void* dst;           // bf16, same layout
  const int* cu;       // null for the dense layout; else int32 [B + 1]
  int B, H, L, D;      // L: rows per sequence (dense)
  int total;           // packed: tokens
  int pos_off;         // dense: added to every row's position (queries: Lkv - Lq)
  const int* cu_kv;    // packed queries: the keys' offsets; a sequence's rows are shifted by its Lkv - Lq
  RopeArgs rope;
  unsigned* status;
  cudaStream_t stream;
};

cudaError_t launch_rope_rows(const RopeRowsLaunch& p);

// One thread waits on a barrier nothing arrives on, with the kernels' bounded wait and a limit of limit_ns.
cudaError_t launch_selftest_timeout(unsigned long long limit_ns, unsigned* status, cudaStream_t stream);

}  // namespace attn
