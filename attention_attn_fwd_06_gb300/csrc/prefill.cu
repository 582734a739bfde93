// prefill.cu -- fused attention forward for prefill on the 5th-generation
// tensor cores (tcgen05 MMAs, TMEM accumulators, TMA-fed shared memory).
//
// What it computes: for each query tile Q_i (128 rows), the tiled online
// softmax of "GPU 学习日报 Day 24：Operator Fusion" §3.4 (second listing):
// stream K_j, V_j tiles on chip, S_ij = Q_i K_j^T, keep the running row max
// m and row sum l, rescale the O accumulator, accumulate P V_j, and normalise
// O by l once at the end, so the S matrix never reaches HBM.  The logits are
// scaled by `scale` and causally masked (bottom-right aligned) as in the
// standard chain of the same section; the per-row log-sum-exp is written too.
//
// GB300 design (two 128-row query tiles per CTA; 10 warps at D = 64, 12 at D = 128 where warpgroup 0 -- TMA,
// MMA and two idle warps -- hands registers to the two softmax warpgroups with setmaxnreg):
//  * warp 0 (one lane) issues TMA tile loads: both Q tiles once, then K_j and
//    V_j into two shared-memory rings (128-byte swizzled boxes of 64 columns x
//    128 rows); a K slot is refilled once the S MMAs reading it are done, a V
//    slot once the P V MMAs are, so loads run about two steps ahead;
//  * warp 1 owns the TMEM allocation (512 columns: S_A, S_B, O_A, O_B) and one
//    lane issues every tcgen05.mma: S_t = Q_t K_j^T (both operands from shared
//    memory, fp32 accumulator in TMEM) and O_t += P_t V_j with P read from TMEM
//    (where it overwrote S_t) and V_j as an MN-major operand (no transpose);
//  * warps 2-5 and 6-9 are one softmax group per query tile, one thread per
//    query row = one TMEM lane: load the S row, mask, row max, exp2 on MUFU,
//    row sum, write P as bf16 over S, and rescale the O row in TMEM when the
//    running max rose by more than 8 (log2 units) -- otherwise the stale max
//    is kept, which is exact because O and l share it;
//  * per K/V step the MMA warp issues P_A V_j, S_A(j+1), P_B V_j, S_B(j+1):
//    one tile's softmax runs while the tensor pipe works for the other tile;
//    its one issuing lane shares an SM sub-partition with two softmax warps,
//    so the shared-memory descriptors are built once and each MMA only adds
//    a constant to one 32-bit half;
//  * dense inputs run one persistent CTA per SM over equal-cost work items
//    (causal: a heavy and a light tile pair of one head; otherwise one tile
//    pair); packed sequences launch one CTA per tile pair, heaviest first;
//    the tiles of one head are adjacent in the order, so K/V stay in L2;
//  * with RoPE the queries and keys arrive already rotated from a pass of
//    their own (rope_rows.cu): rotating K tiles where they land would repeat the
//    work for every query tile of the head, and rotating each Q tile where it
//    lands put the rotation on the MMA warp's path at every job start.
//
// Every wait is bounded (common.cuh); on a timeout the CTA records the status,
// drains its in-flight copies and MMAs, frees TMEM and exits.
#include <cmath>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"
#include "tmap.h"

namespace attn {
namespace {

constexpr int BM = 128;  // query rows per tile (TMEM lanes)
constexpr int BN = 128;  // keys per K/V tile
constexpr int NQ = 2;    // query tiles per CTA (ping-pong)
constexpr int kWarpTMA = 0;
constexpr int kWarpMMA = 1;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: p <= 2^8 between rescales

template <int D>
struct Cfg {
  // Warp roles.  D = 64: 10 warps -- TMA, MMA, then a 4-warp softmax group per query tile (warps 2-5, 6-9).
  // D = 128: 12 warps with a register split -- warpgroup 0 holds the TMA and MMA warps (warps 2-3 idle) and
  // lowers its registers, the two softmax warpgroups (warps 4-7, 8-11) raise theirs, so the softmax threads
  // (128 scores, 64 packed P words and the row state each) keep everything in registers.  Measured on the
  // causal 4k workload: 464 -> 444 us; at D = 64 the split was 1 % slower.  Of the splits 96 / 200, 104 / 192
  // and 112 / 184, 104 / 192 is the one with no spills in either part and measured 0.7 % faster than 96 / 200
  // (452 against 455.5 us, two same-box rounds); 56 / 224 starved the MMA warp (+20 %).
  static constexpr bool SPLIT = (D == 128);
  static constexpr int FIRST_SOFTMAX_WARP = SPLIT ? 4 : 2;
  static constexpr int THREADS = 32 * (FIRST_SOFTMAX_WARP + 4 * NQ);
  // Registers per thread: at launch (the host checks the compiled kernel before its first launch), and after
  // the split.  Each SM sub-partition holds one warp of each warpgroup, so the split fits when one warp of
  // each, after the split, needs no more than the three took at launch; the inc then never waits for ever.
  static constexpr int LAUNCH_REGS = 168;
  static constexpr int REGS_LOW = 104;
  static constexpr int REGS_HIGH = 192;
  static_assert(!SPLIT || (THREADS == 3 * 128 && REGS_LOW + NQ * REGS_HIGH <= 3 * LAUNCH_REGS &&
                           REGS_LOW % 8 == 0 && REGS_HIGH % 8 == 0 && REGS_LOW >= 24 && REGS_HIGH <= 256),
                "register split must fit the launch allocation");
  static constexpr int NDB = D / 64;             // 128-byte column blocks per row
  static constexpr int TILE_BYTES = BM * D * 2;  // one Q, K or V tile (BM == BN)
  static constexpr int BLOCK_BYTES = BM * 128;   // one 64-column block of a tile
  static constexpr int NSV = (D == 128) ? 2 : 4;  // V ring depth
  static constexpr int NSK = NSV;                  // K ring depth
  static constexpr int OFF_Q = 0;                // NQ query tiles
  static constexpr int OFF_K = OFF_Q + NQ * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NSK * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_V + NSV * TILE_BYTES;
  // barriers: q_full, q_empty, k_full[NSK], v_full[NSV], k_empty[NSK], v_empty[NSV], s_full[NQ], p_full[NQ],
  // o_done[NQ], drain
  static constexpr int NBAR = 2 + 2 * NSK + 2 * NSV + 3 * NQ + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem address, abort flag
  static constexpr int SMEM_USED = OFF_MISC + 16;
  static constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack to align the base to 1024
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory");
  // One CTA per SM, always: a warp may only touch the TMEM lanes of its SM sub-partition, and the role code
  // takes that to be its CTA-local warp index % 4.  That holds when the CTA is alone on its SM (its warps take
  // hardware slots 0..); a second CTA on the same SM starts at the slot after the first CTA's last warp (measured
  // with 6-warp CTAs: slot 6), which breaks the mapping.  The shared memory a CTA takes rules out a second one.
  static_assert(2 * (SMEM_ALLOC + 1024) > 228 * 1024, "the TMEM lane mapping needs one CTA per SM");
  // TMEM columns: S_t (fp32 128 x 128, P_t bf16 aliased in its first 64 columns), O_t (fp32 128 x D)
  static constexpr uint32_t tm_s(int t) { return (uint32_t)(t * BN); }
  static constexpr uint32_t tm_o(int t) { return (uint32_t)(NQ * BN + t * D); }
  static_assert(NQ * BN + NQ * D <= (int)kTmemCols, "TMEM columns");
  static constexpr uint32_t IDESC_S = tc::idesc_bf16_f32(BM, BN, false);
  static constexpr uint32_t IDESC_O = tc::idesc_bf16_f32(BM, D, true);
};

struct PrefillArgs {
  void* out;
  float* lse;
  const int* cu_q;
  const int* cu_k;
  int B, Hq, Hkv, Lq, Lkv;
  int varlen;
  int causal;
  int out_f32;
  float scale_log2;  // |scale| * log2(e), or 1 when scale == 0 (then `uniform` is set)
  uint32_t idesc_s;  // instruction descriptor of the S MMAs: negates Q when scale < 0, so S * scale_log2 keeps the sign
  int uniform;       // scale == 0: every visible logit is 0 (uniform weights), masked ones -inf
  int ns;            // work items per (sequence, head)
  int single;        // 1: an item is one tile pair; 0: an item is the tile pairs np-1-s and s
  int total_items;   // B * Hq * ns
  int total_q, total_k;  // packed layout: rows of q/out and of k/v
  unsigned* status;
  int fault_skip_arrive; // test hook (see launch_prefill's caller): CTA 0 withholds one P-ready arrival
};

// One job = one pair of 128-row query tiles of one (sequence, head).
struct Job {
  int bs, h, hk;
  int q_start, k_start, Lq_s, Lkv_s;
  int q00;  // first row of the first tile
  int off;  // causal alignment: key j visible to row i iff j <= i + off
  int nt[NQ];
  int n;    // max nt: K/V steps of the job
};

// Work item `item` of one (sequence, head) holds either the tile pairs (np-1-s) and s, np being that
// sequence's number of tile pairs -- on a causal square the two cost the same in total, so equal
// numbers of items per persistent CTA balance -- or (single mode) just tile pair np-1-s.  `half` picks
// the heavy (0) or light (1) pair.  Returns false when the job is empty (past the sequence end, the
// middle pair of an odd count, malformed offsets).
__device__ __forceinline__ bool make_job(const PrefillArgs& a, int item, int half, Job& jb) {
  const int s = item % a.ns;
  const int rest = item / a.ns;
  jb.h = rest % a.Hq;
  jb.bs = rest / a.Hq;
  jb.hk = jb.h / (a.Hq / a.Hkv);
  jb.q_start = 0;
  jb.k_start = 0;
  jb.Lq_s = a.Lq;
  jb.Lkv_s = a.Lkv;
  if (a.varlen) {
    jb.q_start = a.cu_q[jb.bs];
    jb.Lq_s = a.cu_q[jb.bs + 1] - jb.q_start;
    jb.k_start = a.cu_k[jb.bs];
    jb.Lkv_s = a.cu_k[jb.bs + 1] - jb.k_start;
    if (jb.q_start < 0 || jb.Lq_s < 0 || jb.Lq_s > a.Lq || jb.q_start + jb.Lq_s > a.total_q || jb.k_start < 0 ||
        jb.Lkv_s < 0 || jb.k_start + jb.Lkv_s > a.total_k) {
      record_status(a.status, ATTN_ERR_DEVICE_BOUNDS);  // malformed cu_seqlens: touch nothing
      return false;
    }
  }
  const int np = (jb.Lq_s + NQ * BM - 1) / (NQ * BM);
  const int heavy = np - 1 - s;
  int pair;
  if (half == 0) {
    pair = heavy;
  } else {
    if (a.single || s >= heavy) return false;  // the middle pair of an odd count is done by half 0
    pair = s;
  }
  if (pair < 0) return false;
  jb.q00 = pair * NQ * BM;
  jb.off = jb.Lkv_s - jb.Lq_s;
  jb.n = 0;
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    const int q0 = jb.q00 + t * BM;
    int n = 0;
    if (q0 < jb.Lq_s && jb.Lkv_s > 0) {
      if (a.causal) {
        const int last_row = min(q0 + BM - 1, jb.Lq_s - 1);
        const int kmax = min(jb.Lkv_s - 1, last_row + jb.off);
        n = (kmax < 0) ? 0 : kmax / BN + 1;
      } else {
        n = (jb.Lkv_s + BN - 1) / BN;
      }
    }
    jb.nt[t] = n;
    jb.n = max(jb.n, n);
  }
  return true;
}

template <int D>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1)
    prefill_fwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const PrefillArgs a) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Qs = smem + C::OFF_Q;
  uint8_t* Ks = smem + C::OFF_K;
  uint8_t* Vs = smem + C::OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;         // Q tiles free: every S MMA of the job has completed
  uint64_t* k_full = bars + 2;
  uint64_t* v_full = k_full + C::NSK;
  uint64_t* k_empty = v_full + C::NSV;   // K slot free: every S = Q K^T reading it has completed
  uint64_t* v_empty = k_empty + C::NSK;  // V slot free: every P V reading it has completed
  uint64_t* s_full = v_empty + C::NSV;
  uint64_t* p_full = s_full + NQ;
  uint64_t* o_done = p_full + NQ;
  uint64_t* drain = o_done + NQ;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i) {
      const bool is_p = (&bars[i] >= p_full) && (&bars[i] < p_full + NQ);
      mbar_init(&bars[i], is_p ? 128 : 1);
    }
    *abort_flag = 0;
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

  // Every role walks the same job sequence: items blockIdx.x, +gridDim.x, ...; two jobs per item.
  if (warp < C::FIRST_SOFTMAX_WARP) {
  // TMA and MMA warps (and, with the register split, the two idle warps of warpgroup 0): one program point per
  // warpgroup for its register change
  if constexpr (C::SPLIT) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REGS_LOW));
  if (warp == kWarpTMA) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tc::tma_prefetch_desc(&tmq);
      tc::tma_prefetch_desc(&tmk);
      tc::tma_prefetch_desc(&tmv);
      auto issue_q = [&](const Job& jb) {
        const int qhead = a.varlen ? jb.h : jb.bs * a.Hq + jb.h;
        uint32_t qbytes = 0;
#pragma unroll
        for (int t = 0; t < NQ; ++t) qbytes += jb.nt[t] > 0 ? C::TILE_BYTES : 0;
        mbar_arrive_expect_tx(q_full, qbytes);
#pragma unroll
        for (int t = 0; t < NQ; ++t) {
          if (jb.nt[t] == 0) continue;
          const int qrow = jb.q_start + jb.q00 + t * BM;
          for (int db = 0; db < C::NDB; ++db)
            tc::tma_load_3d(Qs + t * C::TILE_BYTES + db * C::BLOCK_BYTES, &tmq, db * 64, a.varlen ? qhead : qrow,
                            a.varlen ? qrow : qhead, q_full);
        }
      };
      // K or V tile j of a job into `slot` of its ring
      auto issue_kv = [&](const CUtensorMap* map, uint8_t* ring, uint64_t* full, int slot, const Job& jb, int j) {
        const int khead = a.varlen ? jb.hk : jb.bs * a.Hkv + jb.hk;
        const int krow = jb.k_start + j * BN;
        mbar_arrive_expect_tx(&full[slot], C::TILE_BYTES);
        for (int db = 0; db < C::NDB; ++db)
          tc::tma_load_3d(ring + slot * C::TILE_BYTES + db * C::BLOCK_BYTES, map, db * 64, a.varlen ? khead : krow,
                          a.varlen ? krow : khead, &full[slot]);
      };
      int ks = 0, vs = 0;  // K and V steps issued (ring positions)
      int qjobs = 0;       // jobs whose Q was loaded
      bool ok = true;
      for (int item = blockIdx.x; ok && item < a.total_items; item += gridDim.x) {
        for (int half = 0; ok && half < 2; ++half) {
          Job jb;
          if (!make_job(a, item, half, jb) || jb.n == 0) continue;
          if (qjobs > 0 && !mbar_wait(q_empty, (qjobs - 1) & 1, a.status, abort_flag)) {
            ok = false;
            break;
          }
          issue_q(jb);
          ++qjobs;
          for (int j = 0; j < jb.n; ++j) {
            // K slots free up after the S MMAs, V slots after the P V MMAs: the two rings refill independently
            if (ks >= C::NSK &&
                !mbar_wait(&k_empty[ks % C::NSK], ((ks / C::NSK) - 1) & 1, a.status, abort_flag)) {
              ok = false;
              break;
            }
            issue_kv(&tmk, Ks, k_full, ks % C::NSK, jb, j);
            ++ks;
            if (vs >= C::NSV &&
                !mbar_wait(&v_empty[vs % C::NSV], ((vs / C::NSV) - 1) & 1, a.status, abort_flag)) {
              ok = false;
              break;
            }
            issue_kv(&tmv, Vs, v_full, vs % C::NSV, jb, j);
            ++vs;
          }
        }
      }
      if (!ok || *abort_flag) {  // let in-flight copies land before shared memory is released
        if (qjobs > 0) mbar_wait(q_full, (qjobs - 1) & 1, a.status, nullptr);
        for (int g = (ks > C::NSK ? ks - C::NSK : 0); g < ks; ++g)
          mbar_wait(&k_full[g % C::NSK], (g / C::NSK) & 1, a.status, nullptr);
        for (int g = (vs > C::NSV ? vs - C::NSV : 0); g < vs; ++g)
          mbar_wait(&v_full[g % C::NSV], (g / C::NSV) & 1, a.status, nullptr);
      }
    }
  } else if (warp == kWarpMMA) {
    // ---------------- MMA issuer: S_A, S_B, then per step PV_A, S_A', PV_B, S_B' ----------------
    if (lane == 0) {
      // Descriptor low halves of the first Q, K and V tiles; every MMA below only adds a constant offset.
      const uint32_t q_lo = tc::sw128_desc_lo(smem_u32(Qs), 16);
      const uint32_t k_lo = tc::sw128_desc_lo(smem_u32(Ks), 16);
      const uint32_t v_lo = tc::sw128_desc_lo(smem_u32(Vs), C::BLOCK_BYTES);
      constexpr uint32_t kHi = tc::sw128_desc_hi(1024);
      constexpr uint32_t kTile16 = C::TILE_BYTES >> 4;
      auto issue_s = [&](int t, int g) {
        const uint32_t qa = q_lo + t * kTile16;
        const uint32_t ka = k_lo + (g % C::NSK) * kTile16;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = ((kk >> 2) * C::BLOCK_BYTES + (kk & 3) * 32) >> 4;
          tc::mma_ss(tbase + C::tm_s(t), tc::desc64(qa + koff, kHi), tc::desc64(ka + koff, kHi), a.idesc_s, kk > 0);
        }
        tc::mma_commit(&s_full[t]);
      };
      auto issue_pv = [&](int t, int g, bool first) {
        const uint32_t va = v_lo + (g % C::NSV) * kTile16;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          tc::mma_ts(tbase + C::tm_o(t), tbase + C::tm_s(t) + kk * 8, tc::desc64(va + kk * (2048 >> 4), kHi),
                     C::IDESC_O, (!first || kk > 0) ? 1u : 0u);
        tc::mma_commit(&o_done[t]);
      };
      int kv = 0, qjobs = 0;
      int ps[NQ] = {};  // P V steps issued per tile (p_full phases consumed)
      bool ok = true;
      for (int item = blockIdx.x; ok && item < a.total_items; item += gridDim.x) {
        for (int half = 0; ok && half < 2; ++half) {
          Job jb;
          if (!make_job(a, item, half, jb) || jb.n == 0) continue;
          const int g0 = kv;
          if (!mbar_wait(q_full, qjobs & 1, a.status, abort_flag) ||
              !mbar_wait(&k_full[g0 % C::NSK], (g0 / C::NSK) & 1, a.status,
                         abort_flag)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          // S_t of the new job may overwrite S_t / P_t: the previous job's P_t V was issued before (in order).
#pragma unroll
          for (int t = 0; t < NQ; ++t)
            if (jb.nt[t] > 0) issue_s(t, g0);
          tc::mma_commit(&k_empty[g0 % C::NSK]);
          if (jb.n == 1) tc::mma_commit(q_empty);
          for (int j = 0; ok && j < jb.n; ++j) {
            const int g = g0 + j;
            const int slot = g % C::NSV;
            if (!mbar_wait(&v_full[slot], (g / C::NSV) & 1, a.status, abort_flag)) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
            bool next_s = false;
#pragma unroll
            for (int t = 0; t < NQ; ++t) {
              if (j >= jb.nt[t]) continue;
              // P_t of step j; the job's first P V overwrites O_t, which the softmax group finished reading
              // (its previous epilogue) before it produced this P
              if (!mbar_wait(&p_full[t], ps[t] & 1, a.status, abort_flag)) {
                ok = false;
                break;
              }
              ++ps[t];
              tc::fence_after_sync();
              issue_pv(t, g, j == 0);
              if (j + 1 < jb.nt[t]) {
                if (!mbar_wait(&k_full[(g + 1) % C::NSK], ((g + 1) / C::NSK) & 1,
                               a.status, abort_flag)) {
                  ok = false;
                  break;
                }
                tc::fence_after_sync();
                issue_s(t, g + 1);  // S_t aliases P_t: issued after P_t V_j, the tensor pipe keeps the order
                next_s = true;
              }
            }
            if (!ok) break;
            tc::mma_commit(&v_empty[slot]);                         // both P V_j issued
            if (next_s) tc::mma_commit(&k_empty[(g + 1) % C::NSK]);  // every S reading K_{j+1} issued
            if (j == jb.n - 2) tc::mma_commit(q_empty);             // the job's last S MMAs are issued
          }
          kv += jb.n;
          ++qjobs;
        }
      }
      // Whatever happened, wait for every MMA issued above before TMEM is released.
      tc::mma_commit(drain);
      mbar_wait(drain, 0, a.status, nullptr);
    }
  }
  } else {
    if constexpr (C::SPLIT) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REGS_HIGH));
    // ---------------- softmax + correction + epilogue: one thread per query row ----------------
    const int t = (warp - C::FIRST_SOFTMAX_WARP) >> 2;  // which query tile of each job this group owns
    const int quarter = warp & 3;                    // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;             // row of the tile == TMEM lane
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const float c = a.scale_log2;
    const uint32_t s_addr = tbase + lane_addr + C::tm_s(t);
    const uint32_t o_addr = tbase + lane_addr + C::tm_o(t);
    int ss = 0;  // S steps of this tile consumed so far (s_full / o_done phases)
    bool ok = true;

    for (int item = blockIdx.x; ok && item < a.total_items; item += gridDim.x) {
      for (int half = 0; ok && half < 2; ++half) {
        Job jb;
        if (!make_job(a, item, half, jb)) continue;
        const int q0 = jb.q00 + t * BM;
        if (q0 >= jb.Lq_s) continue;                    // this tile lies past the sequence end
        const int qi = q0 + row;                         // query index within its sequence
        const int horizon = qi + jb.off;                 // last visible key under the causal mask
        const int my_n = jb.nt[t];
        float m_ref = -INFINITY;                         // running max, scaled log2 units
        float l = 0.f;

        for (int j = 0; j < my_n; ++j) {
          if (!mbar_wait(&s_full[t], ss & 1, a.status, abort_flag)) {
            ok = false;
            break;
          }
          ++ss;
          tc::fence_after_sync();
          uint32_t sr[4][32];
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) tc::tmem_ld32(s_addr + cc * 32, sr[cc]);
          tc::tmem_ld_wait();

          // The mask acts on the scaled logits (scale, then mask): with scale > 0 -- the host makes the factor
          // positive by negating Q in the S MMA when scale < 0 -- a raw -inf stays -inf once scaled.  With
          // scale == 0 every visible logit is 0, so those tiles set visible scores to 0 and masked ones to -inf.
          const int kbase = j * BN;
          const bool need_mask = (kbase + BN > jb.Lkv_s) || (a.causal && kbase + BN - 1 > q0 + jb.off);
          if (need_mask || a.uniform) {
            const int lim = a.causal ? min(jb.Lkv_s - 1, horizon) : (jb.Lkv_s - 1);
            if (a.uniform) {
#pragma unroll
              for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  sr[cc][i] = (kbase + cc * 32 + i > lim) ? __float_as_uint(-INFINITY) : 0u;
            } else {
#pragma unroll
              for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (kbase + cc * 32 + i > lim) sr[cc][i] = __float_as_uint(-INFINITY);
            }
          }
          // row max with three-input max (two new values per instruction), four independent chains
          float mx[4];
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            mx[cc] = __uint_as_float(sr[cc][0]);
#pragma unroll
            for (int i = 1; i < 31; i += 2)
              mx[cc] = max3f(mx[cc], __uint_as_float(sr[cc][i]), __uint_as_float(sr[cc][i + 1]));
            mx[cc] = fmaxf(mx[cc], __uint_as_float(sr[cc][31]));
          }
          const float mt = max3f(mx[0], mx[1], fmaxf(mx[2], mx[3])) * c;
          float alpha = 1.f;
          if (mt > m_ref + kRescaleThreshold) {
            alpha = ex2_approx(m_ref - mt);  // 0 when m_ref is still -inf
            m_ref = mt;
            l *= alpha;
          }
          // p = 2^(s*c - m_ref): exponent arguments and row sums on packed fp32x2 FMAs/adds
          // m_ref stays -inf only while every score so far is -inf (masked); then x = -inf and p = 0 with no
          // special case
          const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
          const float2 c2 = make_float2(c, c), n2 = make_float2(neg, neg);
          float2 rs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
          uint32_t pk[2][32];
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[cc][2 * i]), __uint_as_float(sr[cc][2 * i + 1])),
                                          c2, n2);
              const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
              rs[i & 1] = __fadd2_rn(rs[i & 1], pp);
              pk[cc >> 1][(cc & 1) * 16 + i] = tc::pack_bf16x2(pp.x, pp.y);
            }
          }
          l += (rs[0].x + rs[0].y) + (rs[1].x + rs[1].y);
          // P_j (bf16) overwrites the first 64 columns of S_t
          tc::tmem_st32(s_addr, pk[0]);
          tc::tmem_st32(s_addr + 32, pk[1]);
          // O_t correction.  S_t(j) completing implies P_t V_{j-1} completed (issued before it), so O_t is idle.
          if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t orr[32];
              tc::tmem_ld32(o_addr + cc * 32, orr);
              tc::tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
              tc::tmem_st32(o_addr + cc * 32, orr);
            }
          }
          tc::tmem_st_wait();
          tc::fence_before_sync();
          // (the test hook: one thread of CTA 0 withholds its arrival for tile 0's second P, so the MMA warp's
          // bounded wait for it runs out and the CTA winds down -- no fault, no hang)
          if (!(a.fault_skip_arrive && blockIdx.x == 0 && t == 0 && j == 1 && row == 0)) mbar_arrive(&p_full[t]);
        }
        if (!ok) break;

        // ---------------- epilogue: O / l, lse ----------------
        if (my_n > 0) {
          // the job's last P V: o_done phase ss - 1 (earlier phases completed before S_t(last) did)
          if (!mbar_wait(&o_done[t], (ss - 1) & 1, a.status, abort_flag)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
        }
        const bool store = qi < jb.Lq_s;
        const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
        size_t orow;  // element offset of this row in out
        if (a.varlen)
          orow = ((size_t)(jb.q_start + qi) * a.Hq + jb.h) * D;
        else
          orow = (((size_t)jb.bs * a.Hq + jb.h) * a.Lq + qi) * D;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t orr[32];
          if (my_n > 0) {
            tc::tmem_ld32(o_addr + cc * 32, orr);
            tc::tmem_ld_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) orr[i] = 0u;
          }
          if (store) {
            if (a.out_f32) {
              float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + orow + cc * 32);
#pragma unroll
              for (int v4 = 0; v4 < 8; ++v4)
                dst[v4] = make_float4(__uint_as_float(orr[4 * v4]) * inv_l, __uint_as_float(orr[4 * v4 + 1]) * inv_l,
                                      __uint_as_float(orr[4 * v4 + 2]) * inv_l,
                                      __uint_as_float(orr[4 * v4 + 3]) * inv_l);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + orow + cc * 32);
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4) {
                uint4 w;
                w.x = tc::pack_bf16x2(__uint_as_float(orr[8 * v4 + 0]) * inv_l,
                                      __uint_as_float(orr[8 * v4 + 1]) * inv_l);
                w.y = tc::pack_bf16x2(__uint_as_float(orr[8 * v4 + 2]) * inv_l,
                                      __uint_as_float(orr[8 * v4 + 3]) * inv_l);
                w.z = tc::pack_bf16x2(__uint_as_float(orr[8 * v4 + 4]) * inv_l,
                                      __uint_as_float(orr[8 * v4 + 5]) * inv_l);
                w.w = tc::pack_bf16x2(__uint_as_float(orr[8 * v4 + 6]) * inv_l,
                                      __uint_as_float(orr[8 * v4 + 7]) * inv_l);
                dst[v4] = w;
              }
            }
          }
        }
        if (store && a.lse != nullptr) {
          const float lse = (l > 0.f) ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
          if (a.varlen)
            a.lse[(size_t)(jb.q_start + qi) * a.Hq + jb.h] = lse;
          else
            a.lse[((size_t)jb.bs * a.Hq + jb.h) * a.Lq + qi] = lse;
        }
        // (the O_t reads above completed -- tcgen05.wait::ld -- before this group's next P is published,
        //  which is what the next job's first P V waits for)
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
cudaError_t launch_d(const PrefillLaunch& p) {
  using C = Cfg<D>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(prefill_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    if (C::SPLIT) {
      // the kernel's register split assumes this many registers per thread at launch: refuse to launch a
      // build that compiled to another count rather than let an increase wait for registers that never come
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, prefill_fwd_kernel<D>);
      if (e != cudaSuccess) return e;
      if (fa.numRegs != C::LAUNCH_REGS) return cudaErrorInvalidKernelImage;
    }
    attr_set[dev] = true;
  }
  const bool varlen = p.cu_q != nullptr;
  CUtensorMap tmq, tmk, tmv;
  const uint64_t row_b = (uint64_t)D * 2;
  bool ok;
  if (!varlen) {
    // (d, row, b*H + h): rows of one head are contiguous
    const uint64_t Lk = p.Lkv > 0 ? (uint64_t)p.Lkv : 1;
    const void* kb = p.Lkv > 0 ? p.k : p.q;  // Lkv == 0: never read, any valid map
    const void* vb = p.Lkv > 0 ? p.v : p.q;
    ok = make_tmap_bf16_3d(&tmq, p.q, D, p.Lq, (uint64_t)p.B * p.Hq, row_b, row_b * p.Lq, 64, BM, 1) &&
         make_tmap_bf16_3d(&tmk, kb, D, Lk, (uint64_t)p.B * p.Hkv, row_b, row_b * Lk, 64, BN, 1) &&
         make_tmap_bf16_3d(&tmv, vb, D, Lk, (uint64_t)p.B * p.Hkv, row_b, row_b * Lk, 64, BN, 1);
  } else {
    // (d, h, token): one box = 128 consecutive tokens of one head
    const uint64_t tk = p.total_k > 0 ? (uint64_t)p.total_k : 1;
    const void* kb = p.total_k > 0 ? p.k : p.q;
    const void* vb = p.total_k > 0 ? p.v : p.q;
    const uint64_t hk = p.total_k > 0 ? (uint64_t)p.Hkv : 1;
    ok = make_tmap_bf16_3d(&tmq, p.q, D, p.Hq, p.total_q, row_b, row_b * p.Hq, 64, 1, BM) &&
         make_tmap_bf16_3d(&tmk, kb, D, hk, tk, row_b, row_b * hk, 64, 1, BN) &&
         make_tmap_bf16_3d(&tmv, vb, D, hk, tk, row_b, row_b * hk, 64, 1, BN);
  }
  if (!ok) return cudaErrorInvalidValue;
  PrefillArgs a;
  a.out = p.out;
  a.lse = p.lse;
  a.cu_q = p.cu_q;
  a.cu_k = p.cu_k;
  a.B = p.B;
  a.Hq = p.Hq;
  a.Hkv = p.Hkv;
  a.Lq = p.Lq;
  a.Lkv = p.Lkv;
  a.varlen = varlen ? 1 : 0;
  a.causal = p.causal;
  a.out_f32 = p.out_f32;
  // S * scale in log2 units with a positive factor: a negative scale negates Q inside the S MMA instead (exact),
  // and scale == 0 runs the uniform-weight form (factor 1 on logits the mask pass sets to 0 or -inf)
  a.uniform = (p.scale == 0.f) ? 1 : 0;
  a.scale_log2 = a.uniform ? 1.f : fabsf(p.scale) * kLog2e;
  a.idesc_s = C::IDESC_S | (p.scale < 0.f ? tc::kIdescNegateA : 0u);
  const int npairs = (p.Lq + NQ * BM - 1) / (NQ * BM);
  // Dense inputs: persistent CTAs (one per SM) over equal-cost items -- two mirrored tile pairs when causal,
  // one tile pair otherwise -- so a CTA's start-up is paid once.  Packed sequences differ in cost: one CTA per
  // tile pair, heaviest first, balances better.
  const bool persistent = !varlen;
  const bool mirrored = persistent && p.causal;
  a.single = mirrored ? 0 : 1;
  a.ns = mirrored ? (npairs + 1) / 2 : npairs;
  a.total_q = p.total_q;
  a.total_k = p.total_k;
  a.status = p.status;
  a.fault_skip_arrive = p.fault_skip_arrive;
  const long long items = (long long)p.B * p.Hq * a.ns;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  a.total_items = (int)items;
  // persistent: one CTA per SM (shared memory allows no more); otherwise one CTA per item
  int grid = persistent ? (p.num_sms > 0 ? p.num_sms : 148) : a.total_items;
  if (grid > a.total_items) grid = a.total_items;
  if (grid < 1) grid = 1;
  prefill_fwd_kernel<D><<<grid, C::THREADS, C::SMEM_ALLOC, p.stream>>>(tmq, tmk, tmv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillLaunch& p) {
  if (p.D == 64) return launch_d<64>(p);
  if (p.D == 128) return launch_d<128>(p);
  return cudaErrorNotSupported;
}

}  // namespace attn
