// decode_multi.cu -- decode of several new tokens per sequence (multi-token or
// speculative decode) over a KV cache, on the 5th-generation tensor cores.
//
// What it computes: rows 0..n-1 of sequence b's cache (n = kv_lens[b]) hold
// all of its keys, the Lq new tokens' own keys being the last Lq of them; new
// token t attends to keys 0..n-Lq+t (the causal mask aligned to the
// bottom-right corner, as for prefill), through the tiled online softmax of
// "GPU 学习日报 Day 24：Operator Fusion" §3.4 (second listing).  The decoder
// page ("Оптимизация Decoder Attention для LLM на GPU", "Техника выжимания
// производительности", item 1, and its fused-kernel section) serves several
// query tokens of a step at once, so that the tensor cores have work and each
// K/V block is loaded once for all of them.
//
// GB300 design:
//  * One MMA tile holds every query row that reads one kv head: the GP =
//    Hq/Hkv heads of the group times the Lq tokens, R = GP*Lq <= 128 rows.  In
//    the [B, Hq, Lq, D] layout those rows are contiguous, so one TMA box loads
//    them; rows R..127 of the tile are padding (other heads' queries or zeros)
//    whose results are never stored.
//  * Split-KV by stream-K over 128-key tiles: the tiles of all (sequence, kv
//    head) items are laid end to end and each persistent CTA (one per SM)
//    takes an equal contiguous share, so every CTA streams the same K/V bytes
//    whatever the mix of lengths.  A share covers the tail of one item, whole
//    items and the head of another: only its first and last pieces can be
//    partial.
//  * Warp 0 loads Q once per piece and K_j, V_j into a ring of 128-byte
//    swizzled TMA tiles (3 stages at D = 128); warp 1 issues the tcgen05 MMAs:
//    S_j = Q K_j^T into one of two TMEM buffers, so the next tile's scores are
//    computed while the softmax works on this one, and O += P_j V_j with P read
//    from TMEM where it overwrote S_j; warps 2-5 run the softmax, one thread
//    per row (= TMEM lane), with the lazy O rescale of the prefill kernel.
//  * The last tile of an item is loaded so that it ENDS at key n: it starts at
//    n - 128, its keys below the previous tile's end are masked out, and
//    before key 0 the TMA box reads zeros.  No cache row at or past kv_len is
//    read, so whatever those rows hold cannot reach O through 0 * NaN.
//  * A piece holding a whole item writes O / l and the log-sum-exp directly;
//    otherwise it writes (O, m, l) to its partial slot and the CTA that lands
//    an item's last partial (per-item counter, reset by that CTA) merges them.
//
// Every wait is bounded (common.cuh); on a timeout the CTA records the status,
// drains its in-flight copies and MMAs, frees TMEM and exits.
#include <cmath>

#include "common.cuh"
#include "intdiv.h"
#include "kernels.h"
#include "rope.cuh"
#include "tcgen05.cuh"
#include "tmap.h"

namespace attn {
namespace {

constexpr int BM = 128;  // rows of the query tile (TMEM lanes)
constexpr int BN = 128;  // keys per K/V tile
constexpr int kThreads = 32 * 6;  // TMA warp, MMA warp, four softmax warps
constexpr int kWarpTMA = 0;
constexpr int kWarpMMA = 1;
constexpr int kFirstSoftmaxWarp = 2;
constexpr int kSoftmaxThreads = 128;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: p <= 2^8 between rescales

template <int D>
struct MCfg {
  static constexpr int NDB = D / 64;             // 128-byte column blocks per row
  static constexpr int TILE_BYTES = BM * D * 2;  // a Q, K or V tile (BM == BN)
  static constexpr int BLOCK_BYTES = BM * 128;   // one 64-column block of a tile
  static constexpr int NS = (D == 128) ? 3 : 6;  // K/V ring depth
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NS * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_V + NS * TILE_BYTES;
  // barriers: q_full, q_empty, k_full[NS], v_full[NS], k_empty[NS], v_empty[NS], s_full[2], p_full[2],
  // o_done[2], drain, q_ready
  static constexpr int NBAR = 2 + 4 * NS + 2 + 2 + 2 + 1 + 1 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem address, abort flag, last-partial flag
  static constexpr int SMEM_USED = OFF_MISC + 16;
  static constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack to align the base to 1024
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory");
  // One CTA per SM, always: a warp may only touch the TMEM lanes of its SM sub-partition, and the role code
  // takes that to be its CTA-local warp index % 4.  That holds when the CTA is alone on its SM (its warps take
  // hardware slots 0..); a second CTA on the same SM starts at the slot after the first CTA's last warp (measured
  // with 6-warp CTAs: slot 6), which breaks the mapping.  The shared memory a CTA takes rules out a second one.
  static_assert(2 * (SMEM_ALLOC + 1024) > 228 * 1024, "the TMEM lane mapping needs one CTA per SM");
  // TMEM columns: S buffers 0 and 1 (fp32 128 x 128, P bf16 aliased in their first 64 columns), then O
  static constexpr uint32_t tm_s(int buf) { return (uint32_t)(buf * BN); }
  static constexpr uint32_t TM_O = 2 * BN;
  static_assert(2 * BN + D <= (int)kTmemCols, "TMEM columns");
  static constexpr uint32_t IDESC_S = tc::idesc_bf16_f32(BM, BN, false);
  static constexpr uint32_t IDESC_O = tc::idesc_bf16_f32(BM, D, true);
};

struct MultiArgs {
  const int* kv_lens;
  void* out;
  float* lse;
  float* part_o;       // fp32 [2 * grid][R][D]: unnormalised O of a partial piece
  float* part_ml;      // fp32 [2 * grid][R][2]: (m in log2 units, l); 8-byte aligned
  unsigned* counters;  // [2 + b * Hkv + hk]: partials landed per item; zero between calls
  int B, Hq, Hkv, Lq, Lmax;
  int GP;              // query heads per kv head
  int R;               // GP * Lq real rows of the tile
  int q_box_bytes;     // bytes one Q load brings (all column blocks)
  float scale_log2;    // |scale| * log2(e), or 1 when scale == 0 (then `uniform` is set)
  uint32_t idesc_s;    // instruction descriptor of the S MMAs: negates Q when scale < 0, so S * scale_log2 keeps the sign
  int uniform;         // scale == 0: every visible logit is 0 (uniform weights), masked ones -inf
  int out_f32;
  unsigned* status;
  RopeArgs rope;       // style != 0: the softmax threads rotate the Q tile's rows before the S MMAs
  int fault_skip_arrive;  // test hook: CTA 0 withholds one P-ready arrival (its MMA warp's wait runs out)
};

__device__ __forceinline__ int clamp_len(int len, int Lmax) { return len < 0 ? 0 : (len > Lmax ? Lmax : len); }
__device__ __forceinline__ int tiles_of(int n) { return (n + BN - 1) / BN; }

// One piece of work: tiles [t0, t1) of item (b, hk), whose sequence has n keys in T tiles.
struct Piece {
  int b, hk, n, T, t0, t1;
  int np;      // CTAs holding a piece of the item (1: the whole item is here)
  int slot;    // this CTA's partial slot for the piece
  int cta_lo;  // first CTA holding a piece of the item
  int lo_odd;  // 1 when the item starts inside (not at the start of) cta_lo's share
};

// Cost, in tiles, charged to every item with keys when the tile space is split: its piece-end work
// (epilogue or partial, publish, a possible merge) takes about as long as streaming three K/V tiles.  Sweeps of
// graph-replayed steps, 8-token GQA workload: 1 tile 25.9 us, 2 tiles 25.0-25.3 us, 3 tiles 24.6-24.8 us, 4 tiles
// 25.1 us, 5 and 6 tiles 25.4-25.9 us (same box A/B of 2 and 3, twice: 25.0 / 25.1 against 24.7 / 24.7 us); the
// 131k-key workload is within 0.5 % for 1 to 6.
#ifndef ATTN_DMULTI_ITEM_COST
#define ATTN_DMULTI_ITEM_COST 3
#endif
constexpr int kItemCost = ATTN_DMULTI_ITEM_COST;

// Walks this CTA's share [lo, hi) of the flattened cost space.  Item (b, hk) occupies [start, start + kItemCost
// + T): its tiles are the last T positions, so a share that takes on an item start also takes fewer tiles, and a
// share that falls inside an item's cost-only head takes none of its tiles.  Every role keeps its own copy.
struct Walk {
  long long per, lo, hi, pos, start;  // start: first cost position of the current item
  int b, hk, n, T;
};

// Warp-cooperative set-up: every lane of the calling warp must call it; all lanes get the same walk.
__device__ Walk walk_init(const MultiArgs& a, int lane) {
  Walk w;
  long long part = 0;
  for (int b = lane; b < a.B; b += 32) {
    const int raw = a.kv_lens[b];
    const int n = clamp_len(raw, a.Lmax);
    if (raw != n && blockIdx.x == 0) record_status(a.status, ATTN_ERR_DEVICE_BOUNDS);
    part += n > 0 ? tiles_of(n) + kItemCost : 0;
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
  const long long W = part * a.Hkv;
  const long long G = gridDim.x;
  w.per = floor_div(W + G - 1, G);
  if (w.per < 1) w.per = 1;
  w.lo = (long long)blockIdx.x * w.per;
  w.hi = min(w.lo + w.per, W);
  w.pos = w.lo;
  w.b = 0;
  w.hk = 0;
  w.n = 0;
  w.T = 0;
  w.start = 0;
  if (w.lo >= w.hi) {
    w.pos = w.hi;
    return w;
  }
  // find the sequence holding cost position lo: prefix sums of Hkv * (tiles + kItemCost), 32 sequences per step
  long long base = 0;
  for (int c0 = 0; c0 < a.B; c0 += 32) {
    const int b = c0 + lane;
    long long v = 0;
    if (b < a.B) {
      const int n = clamp_len(a.kv_lens[b], a.Lmax);
      v = n > 0 ? (long long)(tiles_of(n) + kItemCost) * a.Hkv : 0;
    }
    long long incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long up = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += up;
    }
    const long long tot = __shfl_sync(0xffffffffu, incl, 31);
    if (base + tot > w.lo) {
      const unsigned hit = __ballot_sync(0xffffffffu, base + incl > w.lo);
      const int src = __ffs(hit) - 1;
      const long long excl = __shfl_sync(0xffffffffu, incl - v, src);
      w.b = c0 + src;
      w.n = clamp_len(a.kv_lens[w.b], a.Lmax);
      w.T = tiles_of(w.n);
      const long long first = base + excl;  // first cost position of sequence w.b
      w.hk = (int)floor_div(w.lo - first, w.T + kItemCost);
      w.start = first + (long long)w.hk * (w.T + kItemCost);
      break;
    }
    base += tot;
  }
  return w;
}

__device__ __forceinline__ bool walk_next(Walk& w, const MultiArgs& a, Piece& p) {
  while (w.pos < w.hi) {
    const long long ts = w.start + kItemCost;  // the item's tiles: cost positions [ts, ts + T)
    const long long s = max(w.pos, ts), e = min(w.hi, ts + w.T);
    const bool has = s < e;
    if (has) {
      p.b = w.b;
      p.hk = w.hk;
      p.n = w.n;
      p.T = w.T;
      p.t0 = (int)(s - ts);
      p.t1 = (int)(e - ts);
      const long long clo = floor_div(ts, w.per);
      const long long chi = floor_div(ts + w.T - 1, w.per);
      p.np = (int)(chi - clo + 1);
      p.cta_lo = (int)clo;
      p.lo_odd = (ts != clo * w.per) ? 1 : 0;
      p.slot = 2 * (int)blockIdx.x + (s == w.lo ? 0 : 1);
    }
    w.pos = w.start + w.T + kItemCost;
    if (w.pos < w.hi) {  // advance to the next item that has keys
      w.start = w.pos;
      if (++w.hk == a.Hkv) {
        w.hk = 0;
        for (++w.b; w.b < a.B; ++w.b) {
          w.n = clamp_len(a.kv_lens[w.b], a.Lmax);
          if (w.n > 0) break;
        }
        if (w.b >= a.B) w.pos = w.hi;  // cannot happen while pos < hi; stop rather than read past kv_lens
        w.T = tiles_of(w.n);
      }
    }
    if (has) return true;
  }
  return false;
}

// Partial slot of the i-th CTA holding a piece of an item.
__device__ __forceinline__ int slot_of(const Piece& p, int i) { return 2 * (p.cta_lo + i) + (i == 0 ? p.lo_odd : 0); }

template <int D>
__device__ __forceinline__ void store_row(const MultiArgs& a, size_t orow, int cc, const uint32_t (&orr)[32],
                                          float inv_l) {
  if (a.out_f32) {
    float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + orow * D + cc * 32);
#pragma unroll
    for (int v4 = 0; v4 < 8; ++v4)
      dst[v4] = make_float4(__uint_as_float(orr[4 * v4]) * inv_l, __uint_as_float(orr[4 * v4 + 1]) * inv_l,
                            __uint_as_float(orr[4 * v4 + 2]) * inv_l, __uint_as_float(orr[4 * v4 + 3]) * inv_l);
  } else {
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + orow * D + cc * 32);
#pragma unroll
    for (int v4 = 0; v4 < 4; ++v4) {
      uint4 w;
      w.x = tc::pack_bf16x2(__uint_as_float(orr[8 * v4 + 0]) * inv_l, __uint_as_float(orr[8 * v4 + 1]) * inv_l);
      w.y = tc::pack_bf16x2(__uint_as_float(orr[8 * v4 + 2]) * inv_l, __uint_as_float(orr[8 * v4 + 3]) * inv_l);
      w.z = tc::pack_bf16x2(__uint_as_float(orr[8 * v4 + 4]) * inv_l, __uint_as_float(orr[8 * v4 + 5]) * inv_l);
      w.w = tc::pack_bf16x2(__uint_as_float(orr[8 * v4 + 6]) * inv_l, __uint_as_float(orr[8 * v4 + 7]) * inv_l);
      dst[v4] = w;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    decode_multi_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const MultiArgs a) {
  using C = MCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Qs = smem + C::OFF_Q;
  uint8_t* Ks = smem + C::OFF_K;
  uint8_t* Vs = smem + C::OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;         // Q free: every S MMA of the piece has completed
  uint64_t* k_full = bars + 2;
  uint64_t* v_full = k_full + C::NS;
  uint64_t* k_empty = v_full + C::NS;   // K slot free: the S MMA reading it has completed
  uint64_t* v_empty = k_empty + C::NS;  // V slot free: the P V MMA reading it has completed
  uint64_t* s_full = v_empty + C::NS;   // [2] per S buffer
  uint64_t* p_full = s_full + 2;        // [2] per S buffer (128 arrivals)
  uint64_t* o_done = p_full + 2;        // [2] P V of even / odd tiles completed
  uint64_t* drain = o_done + 2;
  uint64_t* q_ready = drain + 1;        // with RoPE: the piece's Q rows are rotated (128 arrivals)
  uint64_t* merge_bar = q_ready + 1;    // an item's partials copied into the idle K/V ring for its merge
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (warp == kWarpTMA && lane == 0) {
    // the tensor maps are fetched while the set-up and the kv_lens read run
    tc::tma_prefetch_desc(&tmq);
    tc::tma_prefetch_desc(&tmk);
    tc::tma_prefetch_desc(&tmv);
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i) {
      const bool many = ((&bars[i] >= p_full) && (&bars[i] < p_full + 2)) || &bars[i] == q_ready;
      mbar_init(&bars[i], many ? kSoftmaxThreads : 1);
    }
    *abort_flag = 0;
    *last_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMMA) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tmem_slot;

  Walk walk = walk_init(a, lane);  // every warp, all lanes
  Piece pc;

  if (warp == kWarpTMA) {
    // ---------------- TMA producer ----------------
    // A piece's Q load must wait until every S MMA of the previous piece has completed (one Q buffer), but its
    // K/V tiles need only free ring slots: they are issued as soon as slots free up, and the Q load goes out
    // from inside the slot waits the moment the previous piece releases the buffer, so a piece boundary does
    // not drain the ring.
    if (lane == 0) {
      const uint64_t kv_policy = l2_policy_evict_first();  // K/V are read once
      int kv = 0;        // K/V tiles issued (ring position)
      int q_issued = 0;  // Q loads issued (one per piece)
      bool q_pending = false;
      int q_row = 0;     // first q row of the piece whose Q is pending
      bool ok = true;
      auto issue_q = [&]() {
        mbar_arrive_expect_tx(q_full, (uint32_t)a.q_box_bytes);
        for (int db = 0; db < C::NDB; ++db) tc::tma_load_3d(Qs + db * C::BLOCK_BYTES, &tmq, db * 64, q_row, 0, q_full);
        ++q_issued;
        q_pending = false;
      };
      auto poll_q = [&]() {
        if (q_pending && (q_issued == 0 || mbar_try_wait(q_empty, (q_issued - 1) & 1))) issue_q();
      };
      // Bounded wait on a ring barrier that keeps issuing the pending Q load when it becomes possible.
      auto wait_slot = [&](uint64_t* bar, uint32_t parity) -> bool {
        const uint64_t t0 = globaltimer_ns();
        while (true) {
          poll_q();
          if (mbar_try_wait(bar, parity)) return true;
          if (*abort_flag) return false;
          if (globaltimer_ns() - t0 > kWaitLimitNs) {
            record_status(a.status, ATTN_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
            return false;
          }
        }
      };
      while (ok && walk_next(walk, a, pc)) {
        if (q_pending) {  // the previous piece's Q is still waiting for the buffer: it goes first
          if (!mbar_wait(q_empty, (q_issued - 1) & 1, a.status, abort_flag)) {
            ok = false;
            break;
          }
          issue_q();
        }
        q_row = (pc.b * a.Hq + pc.hk * a.GP) * a.Lq;
        q_pending = true;
        poll_q();
        const int khead = pc.b * a.Hkv + pc.hk;
        for (int tt = pc.t0; tt < pc.t1; ++tt) {
          const int slot = kv % C::NS;
          const int krow = (tt == pc.T - 1) ? pc.n - BN : tt * BN;  // the last tile ends at key n
          if (kv >= C::NS && !wait_slot(&k_empty[slot], ((kv / C::NS) - 1) & 1)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&k_full[slot], C::TILE_BYTES);
          for (int db = 0; db < C::NDB; ++db)
            tc::tma_load_3d_hint(Ks + slot * C::TILE_BYTES + db * C::BLOCK_BYTES, &tmk, db * 64, krow, khead,
                                 &k_full[slot], kv_policy);
          if (kv >= C::NS && !wait_slot(&v_empty[slot], ((kv / C::NS) - 1) & 1)) {
            mbar_wait(&k_full[slot], (kv / C::NS) & 1, a.status, nullptr);  // K is in flight: let it land
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&v_full[slot], C::TILE_BYTES);
          for (int db = 0; db < C::NDB; ++db)
            tc::tma_load_3d_hint(Vs + slot * C::TILE_BYTES + db * C::BLOCK_BYTES, &tmv, db * 64, krow, khead,
                                 &v_full[slot], kv_policy);
          ++kv;
        }
      }
      if (ok && q_pending) {
        if (mbar_wait(q_empty, (q_issued - 1) & 1, a.status, abort_flag)) issue_q();
      }
      if (*abort_flag) {  // let in-flight copies land before shared memory is released
        if (q_issued > 0) mbar_wait(q_full, (q_issued - 1) & 1, a.status, nullptr);
        for (int g = (kv > C::NS ? kv - C::NS : 0); g < kv; ++g) {
          mbar_wait(&k_full[g % C::NS], (g / C::NS) & 1, a.status, nullptr);
          mbar_wait(&v_full[g % C::NS], (g / C::NS) & 1, a.status, nullptr);
        }
      }
    }
  } else if (warp == kWarpMMA) {
    // ---------------- MMA issuer: S_0, S_1, then per tile P_j V_j, S_{j+2} ----------------
    if (lane == 0) {
      auto issue_s = [&](int buf, int kslot) {
        const uint32_t q_addr = smem_u32(Qs);
        const uint32_t k_addr = smem_u32(Ks + kslot * C::TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * C::BLOCK_BYTES + (kk & 3) * 32;
          tc::mma_ss(tbase + C::tm_s(buf), tc::smem_desc_sw128(q_addr + koff, 16, 1024),
                     tc::smem_desc_sw128(k_addr + koff, 16, 1024), a.idesc_s, kk > 0);
        }
        tc::mma_commit(&s_full[buf]);
        tc::mma_commit(&k_empty[kslot]);
      };
      auto issue_pv = [&](int buf, int vslot, bool first) {
        const uint32_t v_addr = smem_u32(Vs + vslot * C::TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          tc::mma_ts(tbase + C::TM_O, tbase + C::tm_s(buf) + kk * 8,
                     tc::smem_desc_sw128(v_addr + kk * 2048, C::BLOCK_BYTES, 1024), C::IDESC_O,
                     (!first || kk > 0) ? 1u : 0u);
      };
      int g = 0;   // tiles processed before the current piece (global tile index)
      int qj = 0;
      bool ok = true;
      while (ok && walk_next(walk, a, pc)) {
        const int nt = pc.t1 - pc.t0;
        // the piece's Q: landed, and with RoPE rotated by the softmax threads
        if (!mbar_wait(a.rope.style != 0 ? q_ready : q_full, qj & 1, a.status, abort_flag)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        // The first two S of the piece: their buffers were freed by P V MMAs issued before (in order).
        for (int i = 0; i < nt && i < 2; ++i) {
          const int gi = g + i;
          if (!mbar_wait(&k_full[gi % C::NS], (gi / C::NS) & 1, a.status, abort_flag)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          issue_s(gi & 1, gi % C::NS);
        }
        if (!ok) break;
        if (nt <= 2) tc::mma_commit(q_empty);
        for (int i = 0; i < nt; ++i) {
          const int gi = g + i;
          const int buf = gi & 1;
          const int slot = gi % C::NS;
          if (!mbar_wait(&v_full[slot], (gi / C::NS) & 1, a.status, abort_flag) ||
              !mbar_wait(&p_full[buf], (gi >> 1) & 1, a.status, abort_flag)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          // the piece's first P V overwrites O, which the softmax finished reading (its previous epilogue)
          // before it produced this P
          issue_pv(buf, slot, i == 0);
          tc::mma_commit(&o_done[buf]);
          tc::mma_commit(&v_empty[slot]);
          if (i + 2 < nt) {
            const int gn = gi + 2;
            if (!mbar_wait(&k_full[gn % C::NS], (gn / C::NS) & 1, a.status, abort_flag)) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
            issue_s(buf, gn % C::NS);  // S buffer `buf` held P_gi: issued after P_gi V, the pipe keeps the order
            if (i + 2 == nt - 1) tc::mma_commit(q_empty);  // the piece's last S is issued
          }
        }
        g += nt;
        ++qj;
      }
      // Whatever happened, wait for every MMA issued above before TMEM is released.
      tc::mma_commit(drain);
      mbar_wait(drain, 0, a.status, nullptr);
    }
  } else {
    // ---------------- softmax, correction and epilogue: one thread per tile row ----------------
    const int sw = warp - kFirstSoftmaxWarp;  // 0..3
    const int quarter = warp & 3;              // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;       // tile row == TMEM lane
    const int stid = sw * 32 + lane;           // 0..127 among the softmax threads
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const uint32_t o_addr = tbase + lane_addr + C::TM_O;
    const float c = a.scale_log2;
    const int t_row = row % a.Lq;  // which new token this row is (padding rows: meaningless)
    int g = 0;
    int sp = 0;  // pieces seen (q_full / q_ready phases)
    bool ok = true;

    // After a failed wait the softmax threads keep walking their pieces without touching TMEM or waiting, so
    // all of them still pass the same named barriers (a barrier cannot time out).
    while (walk_next(walk, a, pc)) {
      const int nt = pc.t1 - pc.t0;
      const int horizon = pc.n - a.Lq + t_row;  // last key this row sees
      float m_ref = -INFINITY;                  // running max, scaled log2 units
      float l = 0.f;
      if (a.rope.style != 0) {
        // Rotate this thread's query row to its position n - Lq + t (rows that see no key stay as they are),
        // then hand the tile to the MMA warp.
        if (ok) ok = mbar_wait(q_full, sp & 1, a.status, abort_flag);
        if (ok && row < a.R && horizon >= 0) {
          const size_t off = (size_t)horizon * (D / 2);
          rope_rotate_row_sw128<D>(Qs, C::BLOCK_BYTES, row, a.rope.cos + off, a.rope.sin + off, a.rope.style);
        }
        fence_proxy_async_smem();  // the rotated rows are read by the tensor cores (async proxy)
        mbar_arrive(q_ready);
      }
      ++sp;
      for (int i = 0; ok && i < nt; ++i) {
        const int gi = g + i;
        const int buf = gi & 1;
        const int tt = pc.t0 + i;
        if (!mbar_wait(&s_full[buf], (gi >> 1) & 1, a.status, abort_flag)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t s_addr = tbase + lane_addr + C::tm_s(buf);
        uint32_t sr[4][32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tc::tmem_ld32(s_addr + cc * 32, sr[cc]);
        tc::tmem_ld_wait();

        const bool last = (tt == pc.T - 1);
        const int ks = last ? pc.n - BN : tt * BN;  // key of column 0
        // The mask acts on the scaled logits (scale, then mask): the factor is positive (a negative scale negates
        // Q in the S MMA), so a raw -inf stays -inf once scaled; with scale == 0 every visible logit is 0.
        if (last || ks + BN - 1 > pc.n - a.Lq || a.uniform) {
          const int lo_key = last ? (pc.T - 1) * BN : 0;  // earlier keys belong to the previous tile
          if (a.uniform) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                const int key = ks + cc * 32 + e;
                sr[cc][e] = (key < lo_key || key > horizon) ? __float_as_uint(-INFINITY) : 0u;
              }
          } else {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                const int key = ks + cc * 32 + e;
                if (key < lo_key || key > horizon) sr[cc][e] = __float_as_uint(-INFINITY);
              }
          }
        }
        float mx[4];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          mx[cc] = __uint_as_float(sr[cc][0]);
#pragma unroll
          for (int e = 1; e < 31; e += 2)
            mx[cc] = max3f(mx[cc], __uint_as_float(sr[cc][e]), __uint_as_float(sr[cc][e + 1]));
          mx[cc] = fmaxf(mx[cc], __uint_as_float(sr[cc][31]));
        }
        const float mt = max3f(mx[0], mx[1], fmaxf(mx[2], mx[3])) * c;
        float alpha = 1.f;
        if (mt > m_ref + kRescaleThreshold) {
          alpha = ex2_approx(m_ref - mt);  // 0 when m_ref is still -inf
          m_ref = mt;
          l *= alpha;
        }
        const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
        const bool live = m_ref != -INFINITY;
        const float2 c2 = make_float2(c, c), n2 = make_float2(neg, neg);
        float2 rs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        uint32_t pk[2][32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 x =
                __ffma2_rn(make_float2(__uint_as_float(sr[cc][2 * e]), __uint_as_float(sr[cc][2 * e + 1])), c2, n2);
            float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            if (!live) pp = make_float2(0.f, 0.f);
            rs[e & 1] = __fadd2_rn(rs[e & 1], pp);
            pk[cc >> 1][(cc & 1) * 16 + e] = tc::pack_bf16x2(pp.x, pp.y);
          }
        }
        l += (rs[0].x + rs[0].y) + (rs[1].x + rs[1].y);
        tc::tmem_st32(s_addr, pk[0]);
        tc::tmem_st32(s_addr + 32, pk[1]);
        if (i > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // O correction: wait for the previous tile's P V.  S_gi completing implies P_{gi-2} V completed (it
          // was issued before S_gi), so the parity wait on that o_done barrier is unambiguous.
          const int gp = gi - 1;
          if (!mbar_wait(&o_done[gp & 1], (gp >> 1) & 1, a.status, abort_flag)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t orr[32];
            tc::tmem_ld32(o_addr + cc * 32, orr);
            tc::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
            tc::tmem_st32(o_addr + cc * 32, orr);
          }
        }
        tc::tmem_st_wait();
        tc::fence_before_sync();
        // (the test hook: one thread of CTA 0 withholds its arrival for the CTA's second tile, so the MMA warp's
        // bounded wait for it runs out and the CTA winds down -- no fault, no hang)
        if (!(a.fault_skip_arrive && blockIdx.x == 0 && gi == 1 && row == 0)) mbar_arrive(&p_full[buf]);
      }
      g += nt;
      if (ok) {
        // the piece's last P V (its completion follows every earlier one's)
        const int gl = g - 1;
        ok = mbar_wait(&o_done[gl & 1], (gl >> 1) & 1, a.status, abort_flag);
        tc::fence_after_sync();
      }

      // ---------------- epilogue ----------------
      const bool real = row < a.R;
      const size_t row0 = (size_t)(pc.b * a.Hq + pc.hk * a.GP) * a.Lq;  // first out row of the item
      if (pc.np == 1) {
        if (!ok) continue;
        const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t orr[32];
          tc::tmem_ld32(o_addr + cc * 32, orr);
          tc::tmem_ld_wait();
          if (real) store_row<D>(a, row0 + row, cc, orr, inv_l);
        }
        if (real && a.lse != nullptr) a.lse[row0 + row] = (l > 0.f) ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
        continue;
      }
      // partial: unnormalised O, m, l into this CTA's slot
      if (ok) {
        const size_t prow = (size_t)pc.slot * a.R + row;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t orr[32];
          tc::tmem_ld32(o_addr + cc * 32, orr);
          tc::tmem_ld_wait();
          if (real) {
            float4* dst = reinterpret_cast<float4*>(a.part_o + prow * D + cc * 32);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              dst[v4] = make_float4(__uint_as_float(orr[4 * v4]), __uint_as_float(orr[4 * v4 + 1]),
                                    __uint_as_float(orr[4 * v4 + 2]), __uint_as_float(orr[4 * v4 + 3]));
          }
        }
        if (real) reinterpret_cast<float2*>(a.part_ml)[prow] = make_float2(m_ref, l);
      }
      // Publish (the barrier orders every softmax thread's stores before thread 0's release atomic); the CTA
      // that lands the item's last partial merges them all.  After a failure nothing is published.
      named_bar_sync(1, kSoftmaxThreads);
      if (stid == 0) {
        int is_last = 0;
        if (*abort_flag == 0) {
          unsigned* ctr = a.counters + 2 + (size_t)pc.b * a.Hkv + pc.hk;
          const unsigned old = atomic_add_acq_rel_gpu(ctr, 1u);
          is_last = (old == (unsigned)pc.np - 1u);
          if (is_last) atomicExch(ctr, 0u);  // re-arm for the next call
        }
        *last_flag = is_last;
      }
      named_bar_sync(1, kSoftmaxThreads);
      if (*last_flag) {
        // Merge: the 128 threads split the item's rows into 32-column chunks; each thread folds the partials of
        // its chunks in slot order with a running max (fixed order: bitwise reproducible).  When this is the
        // CTA's last piece the K/V ring is idle (every load landed and every MMA reading it completed before
        // this epilogue), so the partials come into it with one round of bulk copies; otherwise two partials'
        // loads are in flight at a time.
        constexpr int CPR = D / 32;  // chunks per row
        const uint32_t pbytes = (uint32_t)a.R * D * 4;  // one partial's O
        const uint32_t mlbytes = (uint32_t)a.R * 8;     // its (m, l) rows
        Walk peek = walk;
        Piece pn;
        const bool in_smem = (a.R % 2 == 0) && !walk_next(peek, a, pn) &&
                             (size_t)pc.np * (pbytes + mlbytes) <= (size_t)2 * C::NS * C::TILE_BYTES;
        const float* sm_o = reinterpret_cast<const float*>(Ks);                                // [np][R][D]
        const float2* sm_ml = reinterpret_cast<const float2*>(Ks + (size_t)pc.np * pbytes);  // [np][R]
        bool merge_ok = true;
        if (in_smem) {
          if (stid == 0) {
            mbar_arrive_expect_tx(merge_bar, (uint32_t)pc.np * (pbytes + mlbytes));
            for (int i = 0; i < pc.np; ++i) {
              const size_t prow = (size_t)slot_of(pc, i) * a.R;
              bulk_g2s(Ks + (size_t)i * pbytes, a.part_o + prow * D, pbytes, merge_bar);
              bulk_g2s(Ks + (size_t)pc.np * pbytes + (size_t)i * mlbytes, a.part_ml + prow * 2, mlbytes, merge_bar);
            }
          }
          merge_ok = mbar_wait(merge_bar, 0, a.status, abort_flag);  // at most one such merge per CTA
          // after a failed wait the copies may still be landing: let them, before shared memory is released
          if (!merge_ok) mbar_wait(merge_bar, 0, a.status, nullptr);
        }
        for (int e = stid; merge_ok && e < a.R * CPR; e += kSoftmaxThreads) {
          const int r = e / CPR;
          const int ch = e - r * CPR;
          float M = -INFINITY, L = 0.f;
          float4 acc[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
          auto fold = [&](float2 ml, const float4 (&o)[8]) {
            if (ml.x > M) {  // new running max: rescale what was folded so far (nothing while M is -inf)
              const float sc = (M == -INFINITY) ? 0.f : ex2_approx(M - ml.x);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                acc[j] = make_float4(acc[j].x * sc, acc[j].y * sc, acc[j].z * sc, acc[j].w * sc);
              L *= sc;
              M = ml.x;
            }
            const float w = (ml.x == -INFINITY) ? 0.f : ex2_approx(ml.x - M);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              acc[j].x = fmaf(w, o[j].x, acc[j].x);
              acc[j].y = fmaf(w, o[j].y, acc[j].y);
              acc[j].z = fmaf(w, o[j].z, acc[j].z);
              acc[j].w = fmaf(w, o[j].w, acc[j].w);
            }
            L = fmaf(w, ml.y, L);
          };
          int i = 0;
          if (in_smem) {
            for (; i < pc.np; ++i) {
              const float4* s0 = reinterpret_cast<const float4*>(sm_o + ((size_t)i * a.R + r) * D + ch * 32);
              float4 o0[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) o0[j] = s0[j];
              fold(sm_ml[(size_t)i * a.R + r], o0);
            }
          }
          for (; i + 1 < pc.np; i += 2) {
            const size_t p0 = (size_t)slot_of(pc, i) * a.R + r;
            const size_t p1 = (size_t)slot_of(pc, i + 1) * a.R + r;
            const float2 ml0 = __ldcg(reinterpret_cast<const float2*>(a.part_ml) + p0);
            const float2 ml1 = __ldcg(reinterpret_cast<const float2*>(a.part_ml) + p1);
            const float4* s0 = reinterpret_cast<const float4*>(a.part_o + p0 * D + ch * 32);
            const float4* s1 = reinterpret_cast<const float4*>(a.part_o + p1 * D + ch * 32);
            float4 o0[8], o1[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              o0[j] = __ldcg(s0 + j);
              o1[j] = __ldcg(s1 + j);
            }
            fold(ml0, o0);
            fold(ml1, o1);
          }
          if (i < pc.np) {
            const size_t p0 = (size_t)slot_of(pc, i) * a.R + r;
            const float2 ml0 = __ldcg(reinterpret_cast<const float2*>(a.part_ml) + p0);
            const float4* s0 = reinterpret_cast<const float4*>(a.part_o + p0 * D + ch * 32);
            float4 o0[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) o0[j] = __ldcg(s0 + j);
            fold(ml0, o0);
          }
          const float inv_L = (L > 0.f) ? 1.f / L : 0.f;
          const size_t orow = row0 + r;
          if (a.out_f32) {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + orow * D + ch * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_float4(acc[j].x * inv_L, acc[j].y * inv_L, acc[j].z * inv_L, acc[j].w * inv_L);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + orow * D + ch * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint4 wv;
              wv.x = tc::pack_bf16x2(acc[2 * j].x * inv_L, acc[2 * j].y * inv_L);
              wv.y = tc::pack_bf16x2(acc[2 * j].z * inv_L, acc[2 * j].w * inv_L);
              wv.z = tc::pack_bf16x2(acc[2 * j + 1].x * inv_L, acc[2 * j + 1].y * inv_L);
              wv.w = tc::pack_bf16x2(acc[2 * j + 1].z * inv_L, acc[2 * j + 1].w * inv_L);
              dst[j] = wv;
            }
          }
          if (ch == 0 && a.lse != nullptr) a.lse[orow] = (L > 0.f) ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
      }
      named_bar_sync(1, kSoftmaxThreads);  // last_flag is reused by the next piece
    }
    // Sequences with no keys: O = 0, lse = -inf, spread over the CTAs.
    if (ok) {
      constexpr int VPT = D / 32;
      for (int b = blockIdx.x; b < a.B; b += gridDim.x) {
        if (clamp_len(a.kv_lens[b], a.Lmax) != 0) continue;
        for (int hk = 0; hk < a.Hkv; ++hk) {
          const size_t row0 = (size_t)(b * a.Hq + hk * a.GP) * a.Lq;
          for (int r = sw; r < a.R; r += 4) {
            const size_t orow = row0 + r;
            if (a.out_f32) {
              float* dst = reinterpret_cast<float*>(a.out) + orow * D + lane * VPT;
#pragma unroll
              for (int v = 0; v < VPT; ++v) dst[v] = 0.f;
            } else {
              __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.out) + orow * D + lane * VPT;
#pragma unroll
              for (int v = 0; v < VPT; v += 2) *reinterpret_cast<uint32_t*>(dst + v) = 0u;
            }
            if (lane == 0 && a.lse != nullptr) a.lse[orow] = -INFINITY;
          }
        }
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kWarpMMA) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tbase, kTmemCols);
  }
}

template <int D>
cudaError_t launch_d(const DecodeMultiLaunch& p) {
  using C = MCfg<D>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(decode_multi_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int GP = p.Hq / p.Hkv;
  const int R = GP * p.Lq;
  if (R < 1 || R > BM) return cudaErrorInvalidValue;
  const int qbox = ((R + 7) / 8) * 8;  // whole 8-row swizzle atoms
  const uint64_t row_b = (uint64_t)D * 2;
  const uint64_t qrows = (uint64_t)p.B * p.Hq * p.Lq;
  const uint64_t Lk = p.Lmax > 0 ? (uint64_t)p.Lmax : 1;
  const void* kb = p.Lmax > 0 ? p.kcache : p.q;  // Lmax == 0: never read, any valid map
  const void* vb = p.Lmax > 0 ? p.vcache : p.q;
  CUtensorMap tmq, tmk, tmv;
  // q as rows (b, h, t) of D columns; caches as (d, key, b * Hkv + hk) like dense prefill K/V
  const bool ok = make_tmap_bf16_3d(&tmq, p.q, D, qrows, 1, row_b, row_b * qrows, 64, (uint32_t)qbox, 1) &&
                  make_tmap_bf16_3d(&tmk, kb, D, Lk, (uint64_t)p.B * p.Hkv, row_b, row_b * Lk, 64, BN, 1) &&
                  make_tmap_bf16_3d(&tmv, vb, D, Lk, (uint64_t)p.B * p.Hkv, row_b, row_b * Lk, 64, BN, 1);
  if (!ok) return cudaErrorInvalidValue;
  MultiArgs a;
  a.kv_lens = p.kv_lens;
  a.out = p.out;
  a.lse = p.lse;
  a.part_o = p.part_o;
  a.part_ml = p.part_ml;
  a.counters = p.counters;
  a.B = p.B;
  a.Hq = p.Hq;
  a.Hkv = p.Hkv;
  a.Lq = p.Lq;
  a.Lmax = p.Lmax;
  a.GP = GP;
  a.R = R;
  a.q_box_bytes = qbox * 128 * C::NDB;
  // a positive factor on the logits: a negative scale negates Q in the S MMA (exact); scale == 0 is uniform weights
  a.uniform = (p.scale == 0.f) ? 1 : 0;
  a.scale_log2 = a.uniform ? 1.f : fabsf(p.scale) * kLog2e;
  a.idesc_s = C::IDESC_S | (p.scale < 0.f ? tc::kIdescNegateA : 0u);
  a.out_f32 = p.out_f32;
  a.status = p.status;
  a.rope = p.rope;
  a.fault_skip_arrive = p.fault_skip_arrive;
  decode_multi_kernel<D><<<decode_multi_grid(p.num_sms), kThreads, C::SMEM_ALLOC, p.stream>>>(tmq, tmk, tmv, a);
  return cudaGetLastError();
}

}  // namespace

int decode_multi_grid(int num_sms) { return num_sms > 0 ? num_sms : 148; }

cudaError_t launch_decode_multi(const DecodeMultiLaunch& p) {
  if (p.D == 64) return launch_d<64>(p);
  if (p.D == 128) return launch_d<128>(p);
  return cudaErrorNotSupported;
}

}  // namespace attn
