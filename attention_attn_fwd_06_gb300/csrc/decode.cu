// decode.cu -- single-token decode attention over a KV cache, split along the
// KV sequence, with the log-sum-exp combine fused into the same launch.
//
// What it computes: for each sequence b and query head hq, the new token's
// query against cached keys 0..kv_len[b]-1, softmax, times V ("Оптимизация
// Decoder Attention для LLM на GPU", section on the structure of attention in
// decoding mode).  The KV sequence is cut into `chunk`-key work items processed
// in parallel (Flash-Decoding, "GPU 学习日报 Day 24：Operator Fusion" FAQ Q4);
// each item runs the online-softmax recurrence of that page's §3.4 second
// listing (running max m, running sum l, rescaled O) and yields an
// unnormalised partial (O_i, m_i, l_i); the partials of a row are merged with
// M = max m_i, w_i = 2^(m_i - M), O = sum w_i O_i / sum w_i l_i,
// lse = (M + log2 sum w_i l_i) ln 2.
//
// GB300 design:
//  * Stream-K split: persistent CTAs (three per SM; two with 8 heads per CTA) each take an equal,
//    contiguous slice of the flattened key space of all (b, kv head, head
//    group) rows -- each row also charged a fixed cost for its piece-end
//    work -- so every CTA streams about the same number of bytes whatever the
//    mix of sequence lengths, and there are no waves and no work-queue
//    atomics.  A slice covers the tail of one row, whole rows, and the head of
//    another; only the first and last pieces of a slice can be partial rows.
//    One CTA serves ALL the query heads of its group, so every K/V byte is
//    read from HBM once (the decoder page's fused kernel loads each K/V block
//    once and reuses it for every query of the step).
//  * A producer warp walks the slice and streams K and V rows (contiguous
//    cache, or pages of a paged cache through its block table) (and, on a row
//    piece's first stage, its q vectors) into a shared-memory ring (two to
//    four stages, 64 or 96 KB of K and V) with 1-D bulk copies on the TMA
//    engine (cp.async.bulk, mbarrier completion, an L2 evict-first policy for
//    the K/V rows), running ahead of the consumers across row boundaries.
//  * Consumer warps read 16-byte vectors of K/V from shared memory.  For a
//    K row, D/8 lanes each hold 8 dims; the q.k partial sums of R rows x GP
//    heads are folded across those lanes with a reduce-scatter of warp
//    shuffles (each level halves the values a lane carries), so every lane
//    ends with exactly one finished score.  Scores are in log2 units (q is
//    pre-multiplied by scale*log2(e)); exponentials use ex2.approx; O is only
//    rescaled when some head's running max rises (warp vote).
//  * At the end of a row piece the consumer warps merge their states through
//    shared memory.  A row held by one CTA is written directly.  Otherwise the
//    piece becomes a partial in the CTA's own slot, and the CTA that lands a
//    row's last partial (per-row atomic counter) merges them: no second
//    kernel.  Counters reset themselves; the workspace is zeroed only when it
//    is created.
#include <cfloat>
#include <cmath>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "slice_map.h"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Tuning constants (compile-time overridable), each set by sweeps of graph-replayed steps of the 8 x 4096 GQA
// (contiguous, paged, RoPE) and 131k-key decode workloads:
//  * STAGE_BYTES: K and V bytes per ring stage for 2 or 4 heads per CTA.  16 KB stages (a four-stage ring, the
//    same bytes in flight as two 32 KB stages): 24.0 against 24.7 us on the GQA workload, 25.2 against 26.6 us
//    paged, 24.4 against 25.6 us with RoPE, 203 against 208 us at 131k keys.  (Before the producer's bookkeeping
//    was made cheap and its copies split across lanes, 16 KB stages were within 1 % and slower paged.)
//  * ROW_COST: keys charged to every row with keys when the key space is split -- its piece-end work (warp
//    merge, output or partial, publish, a possible merge of the row) takes about as long as streaming three
//    32-key stages: with 16 KB stages 96 keys measured 23.9 / 24.7 / 24.4 / 202.5 us on those four workloads,
//    128 keys 24.0 / 25.0 / 24.2 / 202.3 us, 64 keys 24.5 / 25.0 / 24.9 / 202.0 us, 192 keys 24.1 / 25.2 / 24.4 /
//    203.0 us;
//  * RANK_W0: the slice weights by launch rank (slice_map.h; 8 and 7: within 1 %; equal slices: 5 % slower).
#ifndef ATTN_DECODE_ROW_COST
#define ATTN_DECODE_ROW_COST 96
#endif
constexpr int kRowCost = ATTN_DECODE_ROW_COST;
#ifndef ATTN_DECODE_STAGE_BYTES
#define ATTN_DECODE_STAGE_BYTES 16384
#endif
template <int D, int GP>
struct DecodeCfg {
  static constexpr int LPR = D / 8;                           // lanes per K/V row (16 B each)
  static constexpr int RPW = 32 / LPR;                        // rows one warp instruction covers
  static constexpr int R = (LPR / GP) > 1 ? (LPR / GP) : 1;   // row instructions per iteration
  static constexpr int KPI = RPW * R;                         // keys per warp iteration
  static constexpr int VPL = R * GP;                          // partial sums per lane before folding
  static_assert(VPL == LPR, "the fold must leave exactly one score per lane");
  // bytes of K and V per stage (GP = 2 or 4: smaller stages, more of them, with the same bytes in flight)
  static constexpr int STAGE_BYTES = (GP == 2 || GP == 4) ? ATTN_DECODE_STAGE_BYTES : 32768;
  static constexpr int SK = STAGE_BYTES / (D * 4);            // keys per stage
  static constexpr int NW = (SK / KPI) < 4 ? (SK / KPI) : 4;  // consumer warps
  static constexpr int KPW = SK / NW;                         // keys per consumer warp per stage
  static constexpr int ITER = KPW / KPI;
  static_assert(ITER * KPI * NW == SK, "stage must split evenly over the consumer warps");
  static constexpr int MINB = (GP >= 8) ? 2 : 3;             // resident CTAs per SM (register budget)
  static constexpr int NS = ((MINB == 3) ? 2 : 3) * 32768 / STAGE_BYTES;  // ring stages (64 or 96 KB of K and V)
  static constexpr int THREADS = 32 * (NW + 1);
  static constexpr int LENS_CACHE = (GP >= 8) ? 64 : 512;    // kv_lens kept in shared memory for the walk
  static constexpr int TILE_ELEMS = SK * D;
  static constexpr int TILE_BYTES = TILE_ELEMS * 2;
  static constexpr int Q_BYTES = GP * D * 2;                  // q of the group's heads (bf16)
  // shared-memory layout (bytes)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NS * TILE_BYTES;
  static constexpr int ROPE_BYTES = 4 * D;                     // cos and sin rows (D/2 fp32 each) of the q position
  static constexpr int OFF_Q = OFF_V + NS * TILE_BYTES;
  static constexpr int OFF_R = OFF_Q + NS * Q_BYTES;          // rope rows per stage
  static constexpr int OFF_BAR = OFF_R + NS * ROPE_BYTES;     // full[NS], empty[NS]
  static constexpr int OFF_INFO = OFF_BAR + 2 * NS * 8;       // StageInfo[NS]
  static constexpr int OFF_P = OFF_INFO + NS * 32;            // pbuf[NW][32]
  static constexpr int OFF_A = OFF_P + NW * 32 * 4;           // abuf[NW][GP]
  static constexpr int OFF_M = OFF_A + NW * GP * 4;           // mbuf[NW][GP]
  static constexpr int OFF_L = OFF_M + NW * GP * 4;           // lbuf[NW][GP]
  static constexpr int OFF_LENS = OFF_L + NW * GP * 4;        // lens[LENS_CACHE]
  static constexpr int OFF_MISC = OFF_LENS + LENS_CACHE * 4;  // abort flag, last-partial flag
  static constexpr int SMEM = OFF_MISC + 16;
  static_assert(NW * GP * D * 4 <= TILE_BYTES, "the piece-end merge parks every warp's O in one K tile");
  static_assert(KPI * NW * ITER == SK && (KPI * D * 2) % 16 == 0, "a warp's first key group: whole 16-byte rows");
  static_assert(MINB * (SMEM + 1024) <= 228 * 1024, "MINB CTAs per SM");
  static_assert(SK / 8 + 1 <= 32, "a stage spans at most 32 pages of the smallest page size (one lane each)");
};

struct StageInfo {
  int b;       // sequence; -1 marks the end of the work
  int hg;      // kv head * ngroups + head group
  int nk;      // keys in this stage
  int flags;   // 1: first stage of a row piece (q rides along), 2: last stage of the piece
  int np;      // CTAs holding a piece of this row (0: empty sequence, 1: whole row here)
  int slot;    // this CTA's partial slot for the piece
  int cta_lo;  // first CTA holding a piece of the row
  int lo_odd;  // slot parity of that first CTA's piece
};

__device__ __forceinline__ int clamp_len(int len, int Lmax) { return len < 0 ? 0 : (len > Lmax ? Lmax : len); }

// Four consecutive outputs starting at element idx (a multiple of 4), as fp32 or bf16.
__device__ __forceinline__ void store_out4(void* out, size_t idx, float4 v, int out_f32) {
  if (out_f32) {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + idx) = v;
  } else {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 w2;
    w2.x = *reinterpret_cast<uint32_t*>(&lo);
    w2.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + idx) = w2;
  }
}

template <int D, int GP>
__global__ void __launch_bounds__(DecodeCfg<D, GP>::THREADS, DecodeCfg<D, GP>::MINB)
    decode_split_kernel(const DecodeLaunch p, const int ngroups, const int group) {
  using C = DecodeCfg<D, GP>;
  extern __shared__ __align__(128) uint8_t smem[];
  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_K);
  __nv_bfloat16* Vs = reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_V);
  uint8_t* Qs = smem + C::OFF_Q;
  float* Rs = reinterpret_cast<float*>(smem + C::OFF_R);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::NS;
  StageInfo* info = reinterpret_cast<StageInfo*>(smem + C::OFF_INFO);
  float* pbuf = reinterpret_cast<float*>(smem + C::OFF_P);
  float* abuf = reinterpret_cast<float*>(smem + C::OFF_A);
  float* mbuf = reinterpret_cast<float*>(smem + C::OFF_M);
  float* lbuf = reinterpret_cast<float*>(smem + C::OFF_L);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  int* lens_s = reinterpret_cast<int*>(smem + C::OFF_LENS);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Hg = p.Hkv * ngroups;  // rows per sequence
  const int cta = blockIdx.x;
  const bool rope_on = p.rope.style != 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::NW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  // The producer's first kv_lens load is issued before the barrier, so its latency overlaps the set-up.
  const int len_first = (warp == C::NW && lane < p.B) ? p.kv_lens[lane] : 0;
  __syncthreads();

  if (warp == C::NW) {
    // ---------------- producer: walk this CTA's slice of the key space ----------------
    // Total keys W = Hg * sum_b len_b (the whole warp sums the lengths).
    long long wsum = 0;
    int nonempty = 0;  // sequences with keys
    for (int b = lane; b < p.B; b += 32) {
      const int raw = (b == lane) ? len_first : p.kv_lens[b];
      const int len = clamp_len(raw, p.Lmax);
      if (raw != len && cta == 0) record_status(p.status, ATTN_ERR_DEVICE_BOUNDS);
      if (b < C::LENS_CACHE) lens_s[b] = len;
      wsum += len;
      nonempty += len > 0 ? 1 : 0;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
      nonempty += __shfl_xor_sync(0xffffffffu, nonempty, off);
    }
    __syncwarp();
    // The whole producer warp walks the slice in lock-step (lane 0 issues the barrier operations and q copies,
    // the lanes split a stage's K/V copies between them and fetch page-table windows for the paged layout).
    auto seq_len = [&](int b) -> int { return b < C::LENS_CACHE ? lens_s[b] : clamp_len(p.kv_lens[b], p.Lmax); };
    const long long W = wsum * Hg;
    // Slices of at least min_keys keys, but never fewer slices than rows with keys (a CTA per row of a short
    // problem rather than one CTA walking many rows); CTAs past the effective grid only handle empty sequences.
    long long geff = floor_div(W + p.min_keys - 1, p.min_keys);
    if (geff < (long long)nonempty * Hg) geff = (long long)nonempty * Hg;
    if (geff > (long long)gridDim.x) geff = gridDim.x;
    if (geff < 1) geff = 1;
    // The split is made in a cost space where every row with keys also costs kRowCost keys' worth of time for
    // its piece-end work (warp merge, output or partial, publish): a row occupies [rs, rs + kRowCost + len),
    // its keys the last len positions, so a slice that takes on a row start also takes fewer keys.  Slices
    // that fall inside a row's cost-only head take no keys of that row.
    const long long Wc = W + (long long)kRowCost * nonempty * Hg;
    const SliceMap sm = make_slice_map(Wc, geff, C::MINB, gridDim.x);
    const long long lo = sm.start(cta);
    const long long hi = sm.start(cta + 1);

    int t = 0;  // stages issued
    bool ok = true;
    const bool paged = p.block_table != nullptr;
    const uint64_t kv_policy = l2_policy_evict_first();  // K/V are read once
    // Paged layout: lane i holds the block-table entry of page (win_base + i) of sequence win_b, as loaded (it is
    // checked where a copy uses it, so the load's latency overlaps whatever the warp does before that).
    int win_b = -1, win_base = 0, my_page = 0;
    // Make the window hold pages [first, last] of sequence b (last - first < 32).
    auto need_pages = [&](int b, int first, int last) {
      if (b == win_b && first >= win_base && last < win_base + 32) return;
      win_b = b;
      win_base = first;
      const int pg = first + lane;
      my_page = 0;
      // only pages that hold keys of the sequence are read: entries past its last page may hold anything, e.g.
      // the -1 a serving engine pads its block table with
      if (pg < p.max_pages && (long long)pg * p.page_size < seq_len(b))
        my_page = p.block_table[(size_t)b * p.max_pages + pg];
    };
    // Copy keys [k0, k0 + nk) of row (b, hkv) to shared memory at dstk (K) and dstv (V).  Contiguous: lane 0 issues
    // the K copy and lane 1 the V copy.  Paged: lane j issues the copies of the stage's page first + j, the part of
    // it the stage holds (a stage of at most 128 keys over pages of at least 8 keys spans at most 17 pages).
    auto copy_keys = [&](int b, int hkv, int k0, int nk, __nv_bfloat16* dstk, __nv_bfloat16* dstv, uint64_t* bar) {
      if (!paged) {
        if (lane < 2) {
          const size_t row0 = ((size_t)b * p.Hkv + hkv) * (size_t)p.Lmax + (size_t)k0;
          const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(lane == 0 ? p.kcache : p.vcache);
          bulk_g2s_hint(lane == 0 ? dstk : dstv, src + row0 * D, (uint32_t)nk * D * 2, bar, kv_policy);
        }
        return;
      }
      const int ps = p.page_size;
      const int first = k0 / ps, last = (k0 + nk - 1) / ps;
      need_pages(b, first, last);
      const int pg = first + lane;
      int page = __shfl_sync(0xffffffffu, my_page, min(pg, last) - win_base);
      if (pg <= last) {
        if (page < 0 || page >= p.num_pages) {
          record_status(p.status, ATTN_ERR_DEVICE_BOUNDS);  // out-of-pool page id: read page 0 instead
          page = 0;
        }
        const int kl = max(k0, pg * ps), kh = min(k0 + nk, (pg + 1) * ps);  // the stage's keys on this page
        const size_t row0 = ((size_t)page * p.Hkv + hkv) * (size_t)ps + (size_t)(kl - pg * ps);
        const uint32_t bytes = (uint32_t)(kh - kl) * D * 2;
        bulk_g2s_hint(dstk + (size_t)(kl - k0) * D, reinterpret_cast<const __nv_bfloat16*>(p.kcache) + row0 * D, bytes,
                      bar, kv_policy);
        bulk_g2s_hint(dstv + (size_t)(kl - k0) * D, reinterpret_cast<const __nv_bfloat16*>(p.vcache) + row0 * D, bytes,
                      bar, kv_policy);
      }
    };
    auto wait_empty = [&](int slot_r) -> bool {
      int okw = 1;
      if (lane == 0) okw = mbar_wait(&empty[slot_r], ((t / C::NS) - 1) & 1, p.status, abort_flag) ? 1 : 0;
      return __shfl_sync(0xffffffffu, okw, 0) != 0;
    };

    // Stream keys [kb, ke) of row (b, hg), whose keys sit at cost positions [ks, ks + len) (first_in_slice: the
    // piece starts this CTA's slice); ke == kb emits one key-less stage (a sequence with no keys).
    auto emit = [&](int b, int hg, int kb, int ke, long long ks, bool first_in_slice) -> bool {
      const int hkv = hg / ngroups;
      const int hq0 = hkv * group + (hg - hkv * ngroups) * GP;
      const __nv_bfloat16* qg = reinterpret_cast<const __nv_bfloat16*>(p.q) + ((size_t)b * p.Hq + hq0) * D;
      const int nkeys = ke - kb;
      const int first = C::SK;  // keys of the piece's first stage
      const int nst = nkeys > 0 ? (nkeys <= first ? 1 : 1 + (nkeys - first + C::SK - 1) / C::SK) : 1;
      int np = 0, slot = 0, cta_lo = 0, lo_odd = 0;  // the piece's merge bookkeeping
      for (int u = 0; u < nst; ++u, ++t) {
        const int slot_r = t % C::NS;
        if (t >= C::NS && !wait_empty(slot_r)) return false;
        const int k0 = (u == 0) ? 0 : first + (u - 1) * C::SK;  // the stage's first key within the piece
        const int nk = nkeys > 0 ? min(u == 0 ? first : C::SK, nkeys - k0) : 0;
        const uint32_t kv_bytes = 2u * (uint32_t)nk * D * 2;
        if (u == 0) {
          // The piece's first copies (K/V, q, and with RoPE the table rows of position kv_len - 1) go out before
          // anything else: their bytes are expected without an arrival, then the bookkeeping below, the stage
          // record and the arrival follow, so the record is written before the phase can complete.
          const bool rope_rows = rope_on && nkeys > 0;
          if (lane == 0) {
            const uint32_t rope_bytes = rope_rows ? (uint32_t)C::ROPE_BYTES : 0u;
            mbar_expect_tx(&full[slot_r], kv_bytes + (uint32_t)C::Q_BYTES + rope_bytes);
          }
          // contiguous K/V go first; a paged stage first loads its block-table window, whose latency the q copy
          // and the bookkeeping below cover, and issues its copies after them
          __nv_bfloat16* const kdst = Ks + slot_r * C::TILE_ELEMS;
          __nv_bfloat16* const vdst = Vs + slot_r * C::TILE_ELEMS;
          if (nk > 0 && !paged) copy_keys(b, hkv, kb, nk, kdst, vdst, &full[slot_r]);
          if (nk > 0 && paged) need_pages(b, kb / p.page_size, (kb + nk - 1) / p.page_size);
          if (lane == 0) {
            bulk_g2s(Qs + slot_r * C::Q_BYTES, qg, C::Q_BYTES, &full[slot_r]);
            if (rope_rows) {
              const size_t pos = (size_t)(seq_len(b) - 1);
              float* rdst = Rs + slot_r * (C::ROPE_BYTES / 4);
              bulk_g2s(rdst, p.rope.cos + pos * (D / 2), D * 2, &full[slot_r]);
              bulk_g2s(rdst + D / 2, p.rope.sin + pos * (D / 2), D * 2, &full[slot_r]);
            }
          }
          if (nk > 0) {
            // Which CTAs hold a piece of this row, and this piece's partial slot.  This CTA's slice holds some of
            // the row's keys [ks, ks + len), so the slices holding its first and last key, c_lo and c_hi, lie on
            // either side of cta; the warp tests 32 slices at a time with starts_by (start is non-decreasing).
            const long long last = ks + seq_len(b) - 1;
            int c_lo = 0, c_hi = cta;
            for (int top = cta;; top -= 32) {  // c_lo: the largest c <= cta with start(c) <= ks
              const unsigned m = __ballot_sync(0xffffffffu, top - lane >= 0 && sm.starts_by(top - lane, ks));
              if (m) {
                c_lo = top - (__ffs(m) - 1);
                break;
              }
            }
            for (int bot = cta + 1;; bot += 32) {  // c_hi: the largest c with start(c) <= last
              const unsigned m = __ballot_sync(0xffffffffu, bot + lane >= sm.g || !sm.starts_by(bot + lane, last));
              if (m) {
                c_hi = bot + (__ffs(m) - 1) - 1;
                break;
              }
            }
            np = c_hi - c_lo + 1;
            cta_lo = c_lo;
            slot = 2 * cta + (first_in_slice ? 0 : 1);
            lo_odd = sm.starts_by(c_lo, ks - 1) ? 1 : 0;  // start(c_lo) < ks
          }
          if (nk > 0 && paged) copy_keys(b, hkv, kb, nk, kdst, vdst, &full[slot_r]);
        }
        if (lane == 0) {
          StageInfo si;
          si.b = b;
          si.hg = hg;
          si.nk = nk;
          si.flags = (u == 0 ? 1 : 0) | (u == nst - 1 ? 2 : 0);
          si.np = np;
          si.slot = slot;
          si.cta_lo = cta_lo;
          si.lo_odd = lo_odd;
          info[slot_r] = si;
          if (u == 0) {
            mbar_arrive(&full[slot_r]);
          } else {
            mbar_arrive_expect_tx(&full[slot_r], kv_bytes);
          }
        }
        if (u > 0 && nk > 0)
          copy_keys(b, hkv, kb + k0, nk, Ks + slot_r * C::TILE_ELEMS, Vs + slot_r * C::TILE_ELEMS, &full[slot_r]);
      }
      return true;
    };

    if (lo < hi) {
      // locate the row whose cost interval holds position `lo`
      long long acc = 0;  // first cost position of sequence b
      int b = 0, len = 0;
      for (; b < p.B; ++b) {
        len = seq_len(b);
        const long long rc = len > 0 ? (long long)len + kRowCost : 0;
        if (acc + (long long)Hg * rc > lo) break;
        acc += (long long)Hg * rc;
      }
      long long rcost = (long long)len + kRowCost;
      int hg = (int)floor_div(lo - acc, rcost);
      long long rs = acc + (long long)hg * rcost;  // cost interval of row (b, hg): [rs, rs + rcost)
      long long pos = lo;
      while (ok && pos < hi) {
        const long long ks = rs + kRowCost;  // its keys: cost positions [ks, ks + len)
        const long long a = max(pos, ks), e = min(hi, ks + len);
        if (a < e) ok = emit(b, hg, (int)(a - ks), (int)(e - ks), ks, a == lo);
        pos = rs + rcost;
        // next row (skip sequences with no keys)
        rs += rcost;
        if (++hg == Hg) {
          hg = 0;
          for (++b; b < p.B; ++b) {
            len = seq_len(b);
            if (len > 0) break;
          }
          rcost = (long long)len + kRowCost;
        }
      }
    }
    // Rows of sequences with no keys: O = 0, lse = -inf, one row per CTA in turn.
    if (nonempty < p.B) {
      for (long long e = cta; ok && e < (long long)p.B * Hg; e += gridDim.x) {
        const int b = (int)floor_div(e, Hg);
        if (seq_len(b) == 0) ok = emit(b, (int)(e - (long long)b * Hg), 0, 0, 0, false);
      }
    }
    if (ok) {
      // end-of-work marker
      const int slot_r = t % C::NS;
      if (t < C::NS || wait_empty(slot_r)) {
        if (lane == 0) {
          info[slot_r].b = -1;
          mbar_arrive(&full[slot_r]);
        }
      }
    }
    if (lane == 0 && *abort_flag) {
      // Let copies already in flight land before the CTA's shared memory is released.
      for (int u = (t > C::NS ? t - C::NS : 0); u < t; ++u)
        mbar_wait(&full[u % C::NS], (u / C::NS) & 1, p.status, nullptr);
    }
    return;
  }

  // ---------------- consumers ----------------
  const int ctid = threadIdx.x;  // 0 .. NW*32-1
  const int nct = C::NW * 32;
  const int sub = lane % C::LPR;  // which 8 dims of a row this lane holds
  const int rw = lane / C::LPR;   // which row of a warp instruction
  const float qscale = p.scale * kLog2e;
  float* pw = pbuf + warp * 32;
  float* aw = abuf + warp * GP;
  // A slot is handed back to the producer once every warp is done with it (the test hook withholds CTA 0's
  // release of its second stage: the producer's bounded wait for that slot then runs out and the CTA winds down,
  // with no fault).
  auto release = [&](int slot, int t) {
    if (lane == 0 && !(p.fault_skip_arrive && cta == 0 && t == 1)) mbar_arrive(&empty[slot]);
  };

  int t = 0;  // stages consumed
  while (true) {
    // ---------------- one row piece; its first stage carries q ----------------
    int slot = t % C::NS;
    if (!mbar_wait(&full[slot], (t / C::NS) & 1, p.status, abort_flag)) break;
    StageInfo si = info[slot];
    if (si.b < 0) break;
    float2 qf[GP][4];     // scaled q, dims 8*sub .. 8*sub+7 as 4 pairs, per head
    float2 o[GP][4];      // O accumulator, same dims
    float m = -INFINITY;  // running max (log2 units) of this lane's head, uniform over the lanes sharing it
    float l = 0.f;        // this lane's share of the running sum
    {
      const __nv_bfloat16* qsm = reinterpret_cast<const __nv_bfloat16*>(Qs + slot * C::Q_BYTES);
      const float* rc = Rs + slot * (C::ROPE_BYTES / 4);  // cos row of the q position; sin row at + D/2
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        float qv[8];
        {
          const uint4 raw = lds128(qsm + g * D + 8 * sub);
          const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) bf16x2_to_f32(w4[j], qv[2 * j], qv[2 * j + 1]);
        }
        if (rope_on && si.nk > 0) {
          // rotate this lane's 8 dims of q to position kv_len - 1 (pair (a, b) -> (a c - b s, b c + a s)), in fp32
          if (p.rope.style == 1) {
            // pairs (i, i + D/2): the partner dims sit in the other half of the row
            const int d0 = 8 * sub;
            const bool low = d0 < D / 2;
            const int i0 = low ? d0 : d0 - D / 2;
            float pv[8];
            const uint4 raw = lds128(qsm + g * D + (low ? d0 + D / 2 : d0 - D / 2));
            const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) bf16x2_to_f32(w4[j], pv[2 * j], pv[2 * j + 1]);
            const float sg = low ? -1.f : 1.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) qv[j] = fmaf(qv[j], rc[i0 + j], sg * pv[j] * rc[D / 2 + i0 + j]);
          } else {
            // pairs (2i, 2i + 1): this lane holds pairs 4 sub .. 4 sub + 3 whole
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float c = rc[4 * sub + k], sn = rc[D / 2 + 4 * sub + k];
              const float a = qv[2 * k], b2 = qv[2 * k + 1];
              qv[2 * k] = fmaf(a, c, -b2 * sn);
              qv[2 * k + 1] = fmaf(b2, c, a * sn);
            }
          }
          // the rotated q is held in bf16, like the tensor the unfused RoPE op would hand to attention
#pragma unroll
          for (int j = 0; j < 8; ++j) qv[j] = __bfloat162float(__float2bfloat16_rn(qv[j]));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          qf[g][j] = make_float2(qv[2 * j] * qscale, qv[2 * j + 1] * qscale);
          o[g][j] = make_float2(0.f, 0.f);
        }
      }
    }
    bool alive = true;
    while (true) {
      const __nv_bfloat16* Kt = Ks + slot * C::TILE_ELEMS;
      const __nv_bfloat16* Vt = Vs + slot * C::TILE_ELEMS;
      const int nk = si.nk;
#pragma unroll 1
      for (int it = 0; it < C::ITER; ++it) {
        // key groups of KPI keys go round-robin over the warps, so a short last stage of a piece still spreads
        const int kb = (it * C::NW + warp) * C::KPI;
        if (kb >= nk) break;  // warp-uniform

        // Load this iteration's K and V rows up front so the V latency hides behind the reductions.
        uint4 kr[C::R], vr[C::R];
#pragma unroll
        for (int r = 0; r < C::R; ++r) {
          const int key = kb + r * C::RPW + rw;
          kr[r] = make_uint4(0, 0, 0, 0);
          vr[r] = make_uint4(0, 0, 0, 0);
          if (key < nk) {
            kr[r] = lds128(Kt + key * D + 8 * sub);
            vr[r] = lds128(Vt + key * D + 8 * sub);
          }
        }
        // S = (scale*log2e) q . k for R rows x GP heads, partial over this lane's 8 dims (packed fp32x2 FMAs)
        float acc[C::VPL];
#pragma unroll
        for (int r = 0; r < C::R; ++r) {
          const uint32_t w4[4] = {kr[r].x, kr[r].y, kr[r].z, kr[r].w};
          float2 kf[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) bf16x2_to_f32(w4[j], kf[j].x, kf[j].y);
#pragma unroll
          for (int g = 0; g < GP; ++g) {
            float2 s2 = __ffma2_rn(qf[g][0], kf[0], make_float2(0.f, 0.f));
#pragma unroll
            for (int j = 1; j < 4; ++j) s2 = __ffma2_rn(qf[g][j], kf[j], s2);
            acc[r * GP + g] = s2.x + s2.y;
          }
        }
        // Reduce-scatter over the LPR lanes of a row: afterwards lane `sub` holds
        // the full score of value index `sub` = (row r = sub / GP, head sub % GP).
#pragma unroll
        for (int mask = C::LPR / 2, n = C::VPL; mask >= 1; mask >>= 1, n >>= 1) {
          const bool up = (sub & mask) != 0;
#pragma unroll
          for (int i = 0; i < n / 2; ++i) {
            const float send = up ? acc[i] : acc[i + n / 2];
            const float keep = up ? acc[i + n / 2] : acc[i];
            acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
          }
        }
        const int my_key = kb + (sub / GP) * C::RPW + rw;
        const float s = (my_key < nk) ? acc[0] : -INFINITY;

        // online softmax for head (sub % GP): max over the lanes that share it
        float tmax = s;
#pragma unroll
        for (int mask = GP; mask < 32; mask <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, mask));
        const float m_new = fmaxf(m, tmax);
        const float alpha = (m_new == -INFINITY) ? 1.f : ex2_approx(m - m_new);
        const float pv = (s == -INFINITY) ? 0.f : ex2_approx(s - m_new);
        l = fmaf(l, alpha, pv);
        m = m_new;

        pw[lane] = pv;
        if (rw == 0 && sub < GP) aw[sub] = alpha;
        __syncwarp();
        if (__any_sync(0xffffffffu, alpha < 1.f)) {
#pragma unroll
          for (int g = 0; g < GP; ++g) {
            const float2 a2 = make_float2(aw[g], aw[g]);
#pragma unroll
            for (int j = 0; j < 4; ++j) o[g][j] = __fmul2_rn(o[g][j], a2);
          }
        }
        // O += P V over the same R rows
#pragma unroll
        for (int r = 0; r < C::R; ++r) {
          const uint32_t w4[4] = {vr[r].x, vr[r].y, vr[r].z, vr[r].w};
          float2 vf[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) bf16x2_to_f32(w4[j], vf[j].x, vf[j].y);
          const float* pr = pw + rw * C::LPR + r * GP;
          float pg[GP];
          if constexpr (GP % 4 == 0) {
#pragma unroll
            for (int g4 = 0; g4 < GP / 4; ++g4) {
              const float4 p4 = reinterpret_cast<const float4*>(pr)[g4];
              pg[4 * g4] = p4.x;
              pg[4 * g4 + 1] = p4.y;
              pg[4 * g4 + 2] = p4.z;
              pg[4 * g4 + 3] = p4.w;
            }
          } else {
#pragma unroll
            for (int g = 0; g < GP; ++g) pg[g] = pr[g];
          }
#pragma unroll
          for (int g = 0; g < GP; ++g) {
            const float2 p2 = make_float2(pg[g], pg[g]);
#pragma unroll
            for (int j = 0; j < 4; ++j) o[g][j] = __ffma2_rn(p2, vf[j], o[g][j]);
          }
        }
        __syncwarp();
      }
      __syncwarp();
      if (si.flags & 2) break;  // the piece's last stage: its slot is released after the merge below
      release(slot, t);
      ++t;
      slot = t % C::NS;
      if (!mbar_wait(&full[slot], (t / C::NS) & 1, p.status, abort_flag)) {
        alive = false;
        break;
      }
      si = info[slot];
    }
    if (!alive) break;

    // ---------------- end of a row piece: merge the consumer warps ----------------
    float lsum = l;
#pragma unroll
    for (int mask = GP; mask < 32; mask <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, mask);
#pragma unroll
    for (int mask = C::LPR; mask < 32; mask <<= 1)
#pragma unroll
      for (int g = 0; g < GP; ++g)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          o[g][j].x += __shfl_xor_sync(0xffffffffu, o[g][j].x, mask);
          o[g][j].y += __shfl_xor_sync(0xffffffffu, o[g][j].y, mask);
        }
    // Each warp parks its O (not yet rescaled) in the K tile of the stage it just finished, scratch until the slot
    // is released below.  With up to 4 heads per CTA a warp's O fits in the K rows of its own first key group,
    // which no other warp reads, so it needs no barrier first; with 8 the warps wait for each other and share the
    // tile.
    constexpr bool kOwnRows = 2 * GP <= C::KPI;
    constexpr int kScrStride = kOwnRows ? C::KPI * D / 2 : GP * D;  // floats between the warps' regions
    float* scr = reinterpret_cast<float*>(Ks + slot * C::TILE_ELEMS);
    if constexpr (!kOwnRows) named_bar_sync(1, nct);
    if (rw == 0) {
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        float4* dst = reinterpret_cast<float4*>(scr + warp * kScrStride + g * D + 8 * sub);
        dst[0] = make_float4(o[g][0].x, o[g][0].y, o[g][1].x, o[g][1].y);
        dst[1] = make_float4(o[g][2].x, o[g][2].y, o[g][3].x, o[g][3].y);
      }
    }
    if (rw == 0 && sub < GP) {
      mbuf[warp * GP + sub] = m;
      lbuf[warp * GP + sub] = lsum;
    }
    named_bar_sync(1, nct);
    const int hkv = si.hg / ngroups;
    const int hq0 = hkv * group + (si.hg - hkv * ngroups) * GP;
    // Output pass over runs of 4 columns: M = max over the warps, each warp's O and sum weighted by 2^(m_w - M) in
    // warp order (bitwise reproducible).  A row held by one CTA is written; otherwise it is this CTA's partial.
    for (int e = ctid; e < GP * D / 4; e += nct) {
      const int g = (4 * e) / D;
      const int d = 4 * e - g * D;
      float M = -INFINITY;
#pragma unroll
      for (int w2 = 0; w2 < C::NW; ++w2) M = fmaxf(M, mbuf[w2 * GP + g]);
      float L = 0.f;
      float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w2 = 0; w2 < C::NW; ++w2) {
        const float mw = mbuf[w2 * GP + g];
        const float wt = (mw == -INFINITY) ? 0.f : ex2_approx(mw - M);
        L = fmaf(wt, lbuf[w2 * GP + g], L);
        const float4 v = reinterpret_cast<const float4*>(scr + w2 * kScrStride + g * D)[d / 4];
        O = make_float4(fmaf(wt, v.x, O.x), fmaf(wt, v.y, O.y), fmaf(wt, v.z, O.z), fmaf(wt, v.w, O.w));
      }
      const size_t bh = (size_t)si.b * p.Hq + hq0 + g;
      if (si.np <= 1) {
        const bool empty_seq = (si.np == 0);
        const float inv = empty_seq ? 0.f : 1.f / L;
        store_out4(p.out, bh * D + d, make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv), p.out_f32);
        if (d == 0 && p.lse != nullptr) p.lse[bh] = empty_seq ? -INFINITY : (M + log2f(L)) * kLn2;
      } else {
        const size_t prow = (size_t)si.slot * GP + g;
        reinterpret_cast<float4*>(p.part_o + prow * D)[d / 4] = O;
        if (d == 0) reinterpret_cast<float2*>(p.part_ml)[prow] = make_float2(M, L);
      }
    }
    fence_proxy_async_smem();  // the scratch stores come before the copy that refills the slot
    // every warp is done with the scratch; for a partial, the barrier also orders every thread's partial stores
    // before thread 0's release fence and atomic below
    named_bar_sync(1, nct);
    release(slot, t);
    ++t;
    if (si.np > 1) {
      // Publish the partial; the CTA that lands a row's last partial merges them all.
      if (ctid == 0) {
        const unsigned ctr = 2u + (unsigned)(si.b * Hg + si.hg);
        // release: the CTA's partial (ordered before this by the barrier) is visible before the count;
        // acquire: when this CTA is the last, the other CTAs' partials are visible to it
        const unsigned old = atomic_add_acq_rel_gpu(&p.counters[ctr], 1u);
        const int is_last = (old == (unsigned)si.np - 1u);
        if (is_last) atomicExch(&p.counters[ctr], 0u);  // re-arm for the next call
        *last_flag = is_last;
      }
      named_bar_sync(1, nct);
      if (*last_flag) {
        // Merge the row's partials: each thread takes a run of 4 columns of one head and folds every partial of
        // the row into it in slot order with a running max (a fixed order: bitwise reproducible), the loads of
        // up to eight partials in flight at a time.  Partial slots of the row: CTA c holds slot 2c (+1 for the
        // first CTA when the row starts inside its slice).
        constexpr int RUNS = GP * D / 4;
        const float2* ml_base = reinterpret_cast<const float2*>(p.part_ml);
        for (int e = ctid; e < RUNS; e += nct) {
          const int g = (e * 4) / D;
          const int d = e * 4 - g * D;
          float M = -INFINITY, L = 0.f;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          auto fold = [&](float2 ml, float4 ov) {
            if (ml.x > M) {  // new running max: rescale what was folded so far (nothing while M is -inf)
              const float sc = (M == -INFINITY) ? 0.f : ex2_approx(M - ml.x);
              acc = make_float4(acc.x * sc, acc.y * sc, acc.z * sc, acc.w * sc);
              L *= sc;
              M = ml.x;
            }
            const float w = (ml.x == -INFINITY) ? 0.f : ex2_approx(ml.x - M);
            acc = make_float4(fmaf(w, ov.x, acc.x), fmaf(w, ov.y, acc.y), fmaf(w, ov.z, acc.z), fmaf(w, ov.w, acc.w));
            L = fmaf(w, ml.y, L);
          };
          auto slot_of = [&](int i) { return 2 * (si.cta_lo + i) + (i == 0 ? si.lo_odd : 0); };
          auto batch = [&](int i, auto n_c) {
            constexpr int N = decltype(n_c)::value;
            float2 ml[N];
            float4 ov[N];
#pragma unroll
            for (int u = 0; u < N; ++u) {
              const size_t prow = (size_t)slot_of(i + u) * GP + g;
              ml[u] = __ldcg(ml_base + prow);
              ov[u] = __ldcg(reinterpret_cast<const float4*>(p.part_o + prow * D + d));
            }
#pragma unroll
            for (int u = 0; u < N; ++u) fold(ml[u], ov[u]);
          };
          int i = 0;
          for (; i + 7 < si.np; i += 8) batch(i, std::integral_constant<int, 8>{});
          for (; i + 1 < si.np; i += 2) batch(i, std::integral_constant<int, 2>{});
          if (i < si.np) batch(i, std::integral_constant<int, 1>{});
          const float inv = 1.f / L;  // L > 0: the row has keys
          const size_t bh = (size_t)si.b * p.Hq + hq0 + g;
          store_out4(p.out, bh * D + d, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv), p.out_f32);
          if (d == 0 && p.lse != nullptr) p.lse[bh] = (M + log2f(L)) * kLn2;
        }
      }
    }
    named_bar_sync(1, nct);  // mbuf/lbuf/last_flag are reused by the next piece
  }
}

template <int D, int GP>
cudaError_t launch_split(const DecodeLaunch& p, int ngroups, int group, int num_sms) {
  using C = DecodeCfg<D, GP>;
  static bool attr_set[64] = {};  // the shared-memory opt-in is per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(decode_split_kernel<D, GP>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  decode_split_kernel<D, GP><<<decode_grid(num_sms, group), C::THREADS, C::SMEM, p.stream>>>(p, ngroups, group);
  return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_gp(const DecodeLaunch& p, int num_sms) {
  const int group = p.Hq / p.Hkv;
  const int gp = decode_heads_per_cta(group);
  const int ngroups = group / gp;
  switch (gp) {
    case 8: return launch_split<D, 8>(p, ngroups, group, num_sms);
    case 4: return launch_split<D, 4>(p, ngroups, group, num_sms);
    case 2: return launch_split<D, 2>(p, ngroups, group, num_sms);
    default: return launch_split<D, 1>(p, ngroups, group, num_sms);
  }
}

}  // namespace

int decode_stage_keys(int D) { return D == 64 ? DecodeCfg<64, 1>::SK : DecodeCfg<128, 1>::SK; }

int decode_heads_per_cta(int group) {
  for (int gp = 8; gp > 1; gp >>= 1)
    if (group % gp == 0) return gp;
  return 1;
}

int decode_grid(int num_sms, int group) {
  const int minb = decode_heads_per_cta(group) >= 8 ? DecodeCfg<128, 8>::MINB : DecodeCfg<128, 4>::MINB;
  return minb * (num_sms > 0 ? num_sms : 148);
}


cudaError_t launch_decode(const DecodeLaunch& p, int num_sms) {
  return (p.D == 64) ? dispatch_gp<64>(p, num_sms) : dispatch_gp<128>(p, num_sms);
}

}  // namespace attn
