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
//  * Stream-K split: persistent CTAs (two per SM) each take an equal,
//    contiguous slice of the flattened key space of all (b, kv head, head
//    group) rows, so every CTA streams the same number of bytes whatever the
//    mix of sequence lengths, and there are no waves and no work-queue
//    atomics.  A slice covers the tail of one row, whole rows, and the head of
//    another; only the first and last pieces of a slice can be partial rows.
//    One CTA serves ALL the query heads of its group, so every K/V byte is
//    read from HBM once (the decoder page's "load each K/V block once, reuse it
//    for all queries of the step").
//  * A producer warp walks the slice and streams K and V rows (and, on a row
//    piece's first stage, its q vectors) into a 3-stage shared-memory ring
//    with 1-D bulk copies on the TMA engine (cp.async.bulk, mbarrier
//    completion), running ahead of the consumers across row boundaries.
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

#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D, int GP>
struct DecodeCfg {
  static constexpr int LPR = D / 8;                           // lanes per K/V row (16 B each)
  static constexpr int RPW = 32 / LPR;                        // rows one warp instruction covers
  static constexpr int R = (LPR / GP) > 1 ? (LPR / GP) : 1;   // row instructions per iteration
  static constexpr int KPI = RPW * R;                         // keys per warp iteration
  static constexpr int VPL = R * GP;                          // partial sums per lane before folding
  static_assert(VPL == LPR, "the fold must leave exactly one score per lane");
  static constexpr int SK = 32768 / (D * 4);                  // keys per stage (16 KB of K + 16 KB of V)
  static constexpr int NW = (SK / KPI) < 4 ? (SK / KPI) : 4;  // consumer warps
  static constexpr int KPW = SK / NW;                         // keys per consumer warp per stage
  static constexpr int ITER = KPW / KPI;
  static_assert(ITER * KPI * NW == SK, "stage must split evenly over the consumer warps");
  static constexpr int NS = 3;                                // ring stages
  static constexpr int THREADS = 32 * (NW + 1);
  static constexpr int TILE_ELEMS = SK * D;
  static constexpr int TILE_BYTES = TILE_ELEMS * 2;
  static constexpr int Q_BYTES = GP * D * 2;                  // q of the group's heads (bf16)
  // shared-memory layout (bytes)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NS * TILE_BYTES;
  static constexpr int OFF_Q = OFF_V + NS * TILE_BYTES;
  static constexpr int OFF_O = OFF_Q + NS * Q_BYTES;          // obuf[GP][D] fp32 (merge)
  static constexpr int OFF_BAR = OFF_O + GP * D * 4;          // full[NS], empty[NS]
  static constexpr int OFF_INFO = OFF_BAR + 2 * NS * 8;       // StageInfo[NS]
  static constexpr int OFF_P = OFF_INFO + NS * 32;            // pbuf[NW][32]
  static constexpr int OFF_A = OFF_P + NW * 32 * 4;           // abuf[NW][GP]
  static constexpr int OFF_M = OFF_A + NW * GP * 4;           // mbuf[NW][GP]
  static constexpr int OFF_L = OFF_M + NW * GP * 4;           // lbuf[NW][GP]
  static constexpr int OFF_MISC = OFF_L + NW * GP * 4;        // abort flag, last-partial flag
  static constexpr int SMEM = OFF_MISC + 16;
  static_assert(SMEM <= 113 * 1024, "two CTAs per SM");
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

template <typename T>
__device__ __forceinline__ void store_out(void* out, size_t idx, float v, int out_f32) {
  if (out_f32)
    reinterpret_cast<float*>(out)[idx] = v;
  else
    reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
}

template <int D, int GP>
__global__ void __launch_bounds__(DecodeCfg<D, GP>::THREADS, 2)
    decode_split_kernel(const DecodeLaunch p, const int ngroups, const int group) {
  using C = DecodeCfg<D, GP>;
  extern __shared__ __align__(128) uint8_t smem[];
  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_K);
  __nv_bfloat16* Vs = reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_V);
  uint8_t* Qs = smem + C::OFF_Q;
  float* obuf = reinterpret_cast<float*>(smem + C::OFF_O);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::NS;
  StageInfo* info = reinterpret_cast<StageInfo*>(smem + C::OFF_INFO);
  float* pbuf = reinterpret_cast<float*>(smem + C::OFF_P);
  float* abuf = reinterpret_cast<float*>(smem + C::OFF_A);
  float* mbuf = reinterpret_cast<float*>(smem + C::OFF_M);
  float* lbuf = reinterpret_cast<float*>(smem + C::OFF_L);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Hg = p.Hkv * ngroups;  // rows per sequence
  const int cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::NW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < GP * D; i += blockDim.x) obuf[i] = 0.f;
  __syncthreads();

  if (warp == C::NW) {
    // ---------------- producer: walk this CTA's slice of the key space ----------------
    // Total keys W = Hg * sum_b len_b (the whole warp sums the lengths).
    long long wsum = 0;
    for (int b = lane; b < p.B; b += 32) {
      const int raw = p.kv_lens[b];
      const int len = clamp_len(raw, p.Lmax);
      if (raw != len && cta == 0) record_status(p.status, ATTN_ERR_DEVICE_BOUNDS);
      wsum += len;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
    if (lane != 0) return;
    const long long W = wsum * Hg;
    // At least min_keys keys per CTA; CTAs past the effective grid only handle empty sequences.
    long long geff = (W + p.min_keys - 1) / p.min_keys;
    if (geff > (long long)gridDim.x) geff = gridDim.x;
    if (geff < 1) geff = 1;
    const long long per = (W + geff - 1) / geff;
    const long long lo = (long long)cta * per;
    const long long hi = min(lo + per, W);

    int t = 0;  // stages issued
    bool ok = true;
    auto emit = [&](int b, int hg, int kb, int ke, int np, int slot, int cta_lo, int lo_odd) -> bool {
      // stream keys [kb, ke) of row (b, hg); ke == kb emits a single key-less stage
      const int hkv = hg / ngroups;
      const int hq0 = hkv * group + (hg - hkv * ngroups) * GP;
      const size_t kv_row0 = ((size_t)b * p.Hkv + hkv) * (size_t)p.Lmax + (size_t)kb;
      const __nv_bfloat16* kg = reinterpret_cast<const __nv_bfloat16*>(p.kcache) + kv_row0 * D;
      const __nv_bfloat16* vg = reinterpret_cast<const __nv_bfloat16*>(p.vcache) + kv_row0 * D;
      const __nv_bfloat16* qg = reinterpret_cast<const __nv_bfloat16*>(p.q) + ((size_t)b * p.Hq + hq0) * D;
      const int nkeys = ke - kb;
      const int nst = nkeys > 0 ? (nkeys + C::SK - 1) / C::SK : 1;
      for (int u = 0; u < nst; ++u, ++t) {
        const int slot_r = t % C::NS;
        if (t >= C::NS && !mbar_wait(&empty[slot_r], ((t / C::NS) - 1) & 1, p.status, abort_flag)) return false;
        const int nk = nkeys > 0 ? min(C::SK, nkeys - u * C::SK) : 0;
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
        const uint32_t bytes = (uint32_t)nk * D * 2;
        mbar_arrive_expect_tx(&full[slot_r], 2 * bytes + (u == 0 ? (uint32_t)C::Q_BYTES : 0u));
        if (nk > 0) {
          bulk_g2s(Ks + slot_r * C::TILE_ELEMS, kg + (size_t)u * C::SK * D, bytes, &full[slot_r]);
          bulk_g2s(Vs + slot_r * C::TILE_ELEMS, vg + (size_t)u * C::SK * D, bytes, &full[slot_r]);
        }
        if (u == 0) bulk_g2s(Qs + slot_r * C::Q_BYTES, qg, C::Q_BYTES, &full[slot_r]);
      }
      return true;
    };

    if (lo < hi) {
      // locate the row holding key `lo`
      long long acc = 0;  // first flattened key of sequence b
      int b = 0, len = 0;
      for (; b < p.B; ++b) {
        len = clamp_len(p.kv_lens[b], p.Lmax);
        if (acc + (long long)Hg * len > lo) break;
        acc += (long long)Hg * len;
      }
      int hg = (int)((lo - acc) / len);
      long long row_start = acc + (long long)hg * len;
      long long pos = lo;
      while (ok && pos < hi) {
        const int kb = (int)(pos - row_start);
        const int ke = (int)min((long long)len, hi - row_start);
        const long long cta_lo = row_start / per;
        const long long cta_hi = (row_start + len - 1) / per;
        const int np = (int)(cta_hi - cta_lo + 1);
        const int slot = 2 * cta + (pos == lo ? 0 : 1);
        const int lo_odd = (row_start != cta_lo * per) ? 1 : 0;
        ok = emit(b, hg, kb, ke, np, slot, (int)cta_lo, lo_odd);
        pos = row_start + ke;
        // next row (skip sequences with no keys)
        row_start += len;
        if (++hg == Hg) {
          hg = 0;
          acc += (long long)Hg * len;
          for (++b; b < p.B; ++b) {
            len = clamp_len(p.kv_lens[b], p.Lmax);
            if (len > 0) break;
          }
          row_start = acc;
        }
      }
    }
    // Sequences with no keys: O = 0, lse = -inf, spread over the CTAs.
    for (int b = cta; ok && b < p.B; b += gridDim.x) {
      if (clamp_len(p.kv_lens[b], p.Lmax) != 0) continue;
      for (int hg = 0; ok && hg < Hg; ++hg) ok = emit(b, hg, 0, 0, 0, 0, 0, 0);
    }
    if (ok) {
      // end-of-work marker
      const int slot_r = t % C::NS;
      if (t < C::NS || mbar_wait(&empty[slot_r], ((t / C::NS) - 1) & 1, p.status, abort_flag)) {
        info[slot_r].b = -1;
        mbar_arrive(&full[slot_r]);
      }
    }
    if (*abort_flag) {
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

  float qf[GP][8];
  float o[GP][8];
  float m = -INFINITY;  // running max (log2 units) of this lane's head, uniform over the lanes sharing it
  float l = 0.f;        // this lane's share of the running sum

  for (int t = 0;; ++t) {
    const int slot = t % C::NS;
    if (!mbar_wait(&full[slot], (t / C::NS) & 1, p.status, abort_flag)) break;
    const StageInfo si = info[slot];
    if (si.b < 0) break;
    const __nv_bfloat16* Kt = Ks + slot * C::TILE_ELEMS;
    const __nv_bfloat16* Vt = Vs + slot * C::TILE_ELEMS;
    if (si.flags & 1) {
      const __nv_bfloat16* qsm = reinterpret_cast<const __nv_bfloat16*>(Qs + slot * C::Q_BYTES);
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        const uint4 raw = lds128(qsm + g * D + 8 * sub);
        const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float lo, hi;
          bf16x2_to_f32(w4[j], lo, hi);
          qf[g][2 * j] = lo * qscale;
          qf[g][2 * j + 1] = hi * qscale;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) o[g][j] = 0.f;
      }
      m = -INFINITY;
      l = 0.f;
    }
    const int nk = si.nk;

#pragma unroll 1
    for (int it = 0; it < C::ITER; ++it) {
      const int kb = warp * C::KPW + it * C::KPI;
      if (kb >= nk) break;  // warp-uniform

      // S = (scale*log2e) q . k for R rows x GP heads, partial over this lane's 8 dims
      float acc[C::VPL];
#pragma unroll
      for (int r = 0; r < C::R; ++r) {
        const int key = kb + r * C::RPW + rw;
        uint4 kr = make_uint4(0, 0, 0, 0);
        if (key < nk) kr = lds128(Kt + key * D + 8 * sub);
        float kf[8];
        bf16x2_to_f32(kr.x, kf[0], kf[1]);
        bf16x2_to_f32(kr.y, kf[2], kf[3]);
        bf16x2_to_f32(kr.z, kf[4], kf[5]);
        bf16x2_to_f32(kr.w, kf[6], kf[7]);
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          float s = 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j) s = fmaf(qf[g][j], kf[j], s);
          acc[r * GP + g] = s;
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
          const float a = aw[g];
#pragma unroll
          for (int j = 0; j < 8; ++j) o[g][j] *= a;
        }
      }
      // O += P V over the same R rows
#pragma unroll
      for (int r = 0; r < C::R; ++r) {
        const int key = kb + r * C::RPW + rw;
        uint4 vr = make_uint4(0, 0, 0, 0);
        if (key < nk) vr = lds128(Vt + key * D + 8 * sub);
        float vf[8];
        bf16x2_to_f32(vr.x, vf[0], vf[1]);
        bf16x2_to_f32(vr.y, vf[2], vf[3]);
        bf16x2_to_f32(vr.z, vf[4], vf[5]);
        bf16x2_to_f32(vr.w, vf[6], vf[7]);
        const float* pr = pw + rw * C::LPR + r * GP;
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          const float pg = pr[g];
#pragma unroll
          for (int j = 0; j < 8; ++j) o[g][j] = fmaf(pg, vf[j], o[g][j]);
        }
      }
      __syncwarp();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);  // this slot's K, V and q are no longer read
    if (!(si.flags & 2)) continue;

    // ---------------- end of a row piece: merge the consumer warps ----------------
    float lsum = l;
#pragma unroll
    for (int mask = GP; mask < 32; mask <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, mask);
    // (o is folded in place: the next piece's first stage re-initialises it)
#pragma unroll
    for (int mask = C::LPR; mask < 32; mask <<= 1)
#pragma unroll
      for (int g = 0; g < GP; ++g)
#pragma unroll
        for (int j = 0; j < 8; ++j) o[g][j] += __shfl_xor_sync(0xffffffffu, o[g][j], mask);
    if (rw == 0 && sub < GP) {
      mbuf[warp * GP + sub] = m;
      lbuf[warp * GP + sub] = lsum;
    }
    named_bar_sync(1, nct);
    // Warps add their rescaled O into obuf one after another (a fixed order keeps results bitwise
    // reproducible); obuf is zero on entry.
#pragma unroll 1
    for (int w = 0; w < C::NW; ++w) {
      if (warp == w && rw == 0) {
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          float M = -INFINITY;
#pragma unroll
          for (int w2 = 0; w2 < C::NW; ++w2) M = fmaxf(M, mbuf[w2 * GP + g]);
          const float mw = mbuf[warp * GP + g];
          const float e = (mw == -INFINITY) ? 0.f : ex2_approx(mw - M);
          float* dst = obuf + g * D + 8 * sub;
#pragma unroll
          for (int j = 0; j < 8; ++j) dst[j] = fmaf(e, o[g][j], dst[j]);
        }
      }
      named_bar_sync(1, nct);
    }
    const int hkv = si.hg / ngroups;
    const int hq0 = hkv * group + (si.hg - hkv * ngroups) * GP;
    for (int idx = ctid; idx < GP * D; idx += nct) {
      const int g = idx / D;
      const int d = idx - g * D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < C::NW; ++w) M = fmaxf(M, mbuf[w * GP + g]);
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < C::NW; ++w) {
        const float mw = mbuf[w * GP + g];
        L = fmaf((mw == -INFINITY) ? 0.f : ex2_approx(mw - M), lbuf[w * GP + g], L);
      }
      const float O = obuf[idx];
      obuf[idx] = 0.f;
      const size_t bh = (size_t)si.b * p.Hq + hq0 + g;
      if (si.np <= 1) {
        const bool empty_seq = (si.np == 0);
        store_out<float>(p.out, bh * D + d, empty_seq ? 0.f : O / L, p.out_f32);
        if (d == 0 && p.lse != nullptr) p.lse[bh] = empty_seq ? -INFINITY : (M + log2f(L)) * kLn2;
      } else {
        const size_t prow = (size_t)si.slot * GP + g;
        p.part_o[prow * D + d] = O;
        if (d == 0) {
          p.part_ml[prow * 2] = M;
          p.part_ml[prow * 2 + 1] = L;
        }
      }
    }
    if (si.np > 1) {
      // Publish the partial; the CTA that lands a row's last partial merges them all.
      __threadfence();
      named_bar_sync(1, nct);
      if (ctid == 0) {
        const unsigned ctr = 2u + (unsigned)(si.b * Hg + si.hg);
        const unsigned old = atomicAdd(&p.counters[ctr], 1u);
        const int is_last = (old == (unsigned)si.np - 1u);
        if (is_last) atomicExch(&p.counters[ctr], 0u);  // re-arm for the next call
        *last_flag = is_last;
      }
      named_bar_sync(1, nct);
      if (*last_flag) {
        __threadfence();
        for (int idx = ctid; idx < GP * D; idx += nct) {
          const int g = idx / D;
          const int d = idx - g * D;
          const size_t bh = (size_t)si.b * p.Hq + hq0 + g;
          // partial slots of the row: CTA c holds slot 2c (+1 for the first CTA when the row
          // starts inside its slice)
          float M = -INFINITY;
#pragma unroll 4
          for (int i = 0; i < si.np; ++i) {
            const int sl = 2 * (si.cta_lo + i) + (i == 0 ? si.lo_odd : 0);
            M = fmaxf(M, __ldcg(p.part_ml + ((size_t)sl * GP + g) * 2));
          }
          float L = 0.f, O = 0.f;
#pragma unroll 4
          for (int i = 0; i < si.np; ++i) {
            const int sl = 2 * (si.cta_lo + i) + (i == 0 ? si.lo_odd : 0);
            const size_t prow = (size_t)sl * GP + g;
            const float w = ex2_approx(__ldcg(p.part_ml + prow * 2) - M);
            L = fmaf(w, __ldcg(p.part_ml + prow * 2 + 1), L);
            O = fmaf(w, __ldcg(p.part_o + prow * D + d), O);
          }
          store_out<float>(p.out, bh * D + d, O / L, p.out_f32);
          if (d == 0 && p.lse != nullptr) p.lse[bh] = (M + log2f(L)) * kLn2;
        }
      }
    }
    named_bar_sync(1, nct);  // mbuf/lbuf/obuf/last_flag are reused by the next piece
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
  decode_split_kernel<D, GP><<<decode_grid(num_sms), C::THREADS, C::SMEM, p.stream>>>(p, ngroups, group);
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

int decode_grid(int num_sms) { return 2 * (num_sms > 0 ? num_sms : 148); }

int decode_heads_per_cta(int group) {
  for (int gp = 8; gp > 1; gp >>= 1)
    if (group % gp == 0) return gp;
  return 1;
}

cudaError_t launch_decode(const DecodeLaunch& p, int num_sms) {
  return (p.D == 64) ? dispatch_gp<64>(p, num_sms) : dispatch_gp<128>(p, num_sms);
}

}  // namespace attn
