// decode.cu -- single-token decode attention over a KV cache, split along the
// KV sequence and merged with a log-sum-exp combine.
//
// What it computes: for each sequence b and query head hq, the new token's
// query against cached keys 0..kv_len[b]-1, softmax, times V ("Оптимизация
// Decoder Attention для LLM на GPU", section on the structure of attention in
// decoding mode).  The KV sequence is cut into `chunk`-key work items processed
// in parallel (Flash-Decoding, "GPU 学习日报 Day 24：Operator Fusion" FAQ Q4);
// each item runs the online-softmax recurrence of that page's §3.4 second
// listing (running max m, running sum l, rescaled O) and writes an
// unnormalised partial (O_i, m_i, l_i); the combine kernel merges them with
// M = max m_i, w_i = 2^(m_i - M), O = sum w_i O_i / sum w_i l_i.
//
// GB300 design:
//  * One CTA serves one (b, kv head, head group, split) item and ALL the query
//    heads of its group, so every K/V byte is read from HBM once (GQA: the
//    decoder page's "load each K/V block once and reuse it for all queries").
//  * A producer warp streams the item's K and V rows into a 3-stage shared
//    memory ring with 1-D bulk copies on the TMA engine (cp.async.bulk,
//    mbarrier completion), so tens of KB per SM are in flight without
//    occupying registers.
//  * Consumer warps read 16-byte vectors of K/V from shared memory.  For a
//    K row, D/8 lanes each hold 8 dims; the q.k partial sums of R rows x GP
//    heads are folded across those lanes with a reduce-scatter of warp
//    shuffles (each level halves the values a lane carries), so every lane
//    ends with exactly one finished score: D/8 - 1 shuffles per D/8 scores.
//  * Scores are kept in log2 units (q is pre-multiplied by scale*log2(e)),
//    exponentials use ex2.approx, and O is only rescaled when some head's
//    running max actually rises (warp vote).
//  * A split that covers a whole sequence writes the final O and lse itself;
//    the combine kernel skips those rows.
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
  // shared-memory layout (bytes)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NS * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_V + NS * TILE_BYTES;     // full[NS], empty[NS]
  static constexpr int OFF_P = OFF_BAR + 2 * NS * 8;          // pbuf[NW][32]
  static constexpr int OFF_A = OFF_P + NW * 32 * 4;           // abuf[NW][GP]
  static constexpr int OFF_M = OFF_A + NW * GP * 4;           // mbuf[NW][GP]
  static constexpr int OFF_L = OFF_M + NW * GP * 4;           // lbuf[NW][GP]
  static constexpr int OFF_ABORT = OFF_L + NW * GP * 4;
  static constexpr int SMEM = OFF_ABORT + 16;
  static_assert(NW * GP * D * 4 <= NS * TILE_BYTES, "merge buffer aliases the K ring");
};

__device__ __forceinline__ int clamp_len(int len, int Lmax) { return len < 0 ? 0 : (len > Lmax ? Lmax : len); }

template <int D, int GP>
__global__ void __launch_bounds__(DecodeCfg<D, GP>::THREADS, 2)
    decode_split_kernel(const DecodeLaunch p, const int ngroups, const int group) {
  using C = DecodeCfg<D, GP>;
  extern __shared__ __align__(128) uint8_t smem[];
  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_K);
  __nv_bfloat16* Vs = reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_V);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::NS;
  float* pbuf = reinterpret_cast<float*>(smem + C::OFF_P);
  float* abuf = reinterpret_cast<float*>(smem + C::OFF_A);
  float* mbuf = reinterpret_cast<float*>(smem + C::OFF_M);
  float* lbuf = reinterpret_cast<float*>(smem + C::OFF_L);
  float* obuf = reinterpret_cast<float*>(smem + C::OFF_K);  // reused after the ring drains
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_ABORT);

  const int split = blockIdx.x;
  const int hkv = blockIdx.y / ngroups;
  const int grp = blockIdx.y - hkv * ngroups;
  const int b = blockIdx.z;

  const int raw_len = p.kv_lens[b];
  const int len = clamp_len(raw_len, p.Lmax);
  if (raw_len != len && split == 0 && blockIdx.y == 0 && threadIdx.x == 0)
    record_status(p.status, ATTN_ERR_DEVICE_BOUNDS);
  const int k0 = split * p.chunk;
  if (k0 >= len) return;  // whole CTA: this split lies past the sequence end
  const int nkeys = min(p.chunk, len - k0);
  const int nst = (nkeys + C::SK - 1) / C::SK;
  const int nsplit_b = (len + p.chunk - 1) / p.chunk;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::NW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const size_t kv_row0 = ((size_t)b * p.Hkv + hkv) * (size_t)p.Lmax + (size_t)k0;
  const __nv_bfloat16* kg = reinterpret_cast<const __nv_bfloat16*>(p.kcache) + kv_row0 * D;
  const __nv_bfloat16* vg = reinterpret_cast<const __nv_bfloat16*>(p.vcache) + kv_row0 * D;
  const int hq0 = hkv * group + grp * GP;

  if (warp == C::NW) {
    // ---------------- producer: one elected lane feeds the ring ----------------
    if (lane == 0) {
      int issued = 0;
      for (int t = 0; t < nst; ++t) {
        const int slot = t % C::NS;
        if (t >= C::NS && !mbar_wait(&empty[slot], ((t / C::NS) - 1) & 1, p.status, abort_flag)) break;
        const int nk = min(C::SK, nkeys - t * C::SK);
        const uint32_t bytes = (uint32_t)nk * D * 2;
        mbar_arrive_expect_tx(&full[slot], 2 * bytes);
        bulk_g2s(Ks + slot * C::TILE_ELEMS, kg + (size_t)t * C::SK * D, bytes, &full[slot]);
        bulk_g2s(Vs + slot * C::TILE_ELEMS, vg + (size_t)t * C::SK * D, bytes, &full[slot]);
        issued = t + 1;
      }
      if (*abort_flag) {
        // Let copies already in flight land before the CTA's shared memory is released.
        for (int t = (issued > C::NS ? issued - C::NS : 0); t < issued; ++t)
          mbar_wait(&full[t % C::NS], (t / C::NS) & 1, p.status, nullptr);
      }
    }
  } else {
    // ---------------- consumers ----------------
    const int sub = lane % C::LPR;  // which 8 dims of a row this lane holds
    const int rw = lane / C::LPR;   // which row of a warp instruction
    const float qscale = p.scale * kLog2e;

    float qf[GP][8];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      const uint4 raw = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.q) +
                                                        ((size_t)b * p.Hq + hq0 + g) * D + 8 * sub);
      const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float lo, hi;
        bf16x2_to_f32(w4[j], lo, hi);
        qf[g][2 * j] = lo * qscale;
        qf[g][2 * j + 1] = hi * qscale;
      }
    }
    float o[GP][8];
#pragma unroll
    for (int g = 0; g < GP; ++g)
#pragma unroll
      for (int j = 0; j < 8; ++j) o[g][j] = 0.f;
    float m = -INFINITY;  // running max (log2 units) of this lane's head, uniform over the lanes sharing it
    float l = 0.f;        // this lane's share of the running sum

    float* pw = pbuf + warp * 32;
    float* aw = abuf + warp * GP;

    for (int t = 0; t < nst; ++t) {
      const int slot = t % C::NS;
      if (!mbar_wait(&full[slot], (t / C::NS) & 1, p.status, abort_flag)) break;
      const int nk = min(C::SK, nkeys - t * C::SK);
      const __nv_bfloat16* Kt = Ks + slot * C::TILE_ELEMS;
      const __nv_bfloat16* Vt = Vs + slot * C::TILE_ELEMS;

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
      if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // Fold this warp's state: l over the lanes sharing a head, O over the rows of a warp instruction.
#pragma unroll
    for (int mask = GP; mask < 32; mask <<= 1) l += __shfl_xor_sync(0xffffffffu, l, mask);
#pragma unroll
    for (int mask = C::LPR; mask < 32; mask <<= 1)
#pragma unroll
      for (int g = 0; g < GP; ++g)
#pragma unroll
        for (int j = 0; j < 8; ++j) o[g][j] += __shfl_xor_sync(0xffffffffu, o[g][j], mask);
    // publish (after every warp has finished reading the ring: see the barrier below)
    named_bar_sync(1, C::NW * 32);
    if (rw == 0) {
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        float* dst = obuf + (warp * GP + g) * D + 8 * sub;
        reinterpret_cast<float4*>(dst)[0] = make_float4(o[g][0], o[g][1], o[g][2], o[g][3]);
        reinterpret_cast<float4*>(dst)[1] = make_float4(o[g][4], o[g][5], o[g][6], o[g][7]);
      }
      if (sub < GP) {
        mbuf[warp * GP + sub] = m;
        lbuf[warp * GP + sub] = l;
      }
    }
  }
  __syncthreads();
  if (*abort_flag) return;

  // ---------------- merge the consumer warps and write ----------------
  const int nthreads = C::NW * 32;
  for (int idx = threadIdx.x; idx < GP * D && threadIdx.x < nthreads; idx += nthreads) {
    const int g = idx / D;
    const int d = idx - g * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::NW; ++w) M = fmaxf(M, mbuf[w * GP + g]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < C::NW; ++w) {
      const float mw = mbuf[w * GP + g];
      const float e = (mw == -INFINITY) ? 0.f : ex2_approx(mw - M);
      L = fmaf(e, lbuf[w * GP + g], L);
      O = fmaf(e, obuf[(w * GP + g) * D + d], O);
    }
    const size_t bh = (size_t)b * p.Hq + hq0 + g;
    if (nsplit_b == 1) {
      const float val = O / L;
      if (p.out_f32)
        reinterpret_cast<float*>(p.out)[bh * D + d] = val;
      else
        reinterpret_cast<__nv_bfloat16*>(p.out)[bh * D + d] = __float2bfloat16_rn(val);
      if (d == 0 && p.lse != nullptr) p.lse[bh] = (M + log2f(L)) * kLn2;
    } else {
      const size_t row = bh * p.nsplit + split;
      p.part_o[row * D + d] = O;
      if (d == 0) {
        p.part_ml[row * 2] = M;
        p.part_ml[row * 2 + 1] = L;
      }
    }
  }
}

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* red) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const float o = __shfl_xor_sync(0xffffffffu, v, off);
    v = is_max ? fmaxf(v, o) : v + o;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = red[0];
  for (int w = 1; w < nw; ++w) v = is_max ? fmaxf(v, red[w]) : v + red[w];
  return v;
}

// One CTA (D threads) per (b, hq): merge the partials of every split of that row.
__global__ void decode_combine_kernel(const DecodeLaunch p) {
  extern __shared__ float wsplit[];
  __shared__ float red[32];
  const int bh = blockIdx.x;
  const int b = bh / p.Hq;
  const int len = clamp_len(p.kv_lens[b], p.Lmax);
  const int n = (len + p.chunk - 1) / p.chunk;
  if (n == 1) return;  // the split pass wrote this row already
  const int d = threadIdx.x;
  const int D = p.D;
  if (n == 0) {
    if (p.out_f32)
      reinterpret_cast<float*>(p.out)[(size_t)bh * D + d] = 0.f;
    else
      reinterpret_cast<__nv_bfloat16*>(p.out)[(size_t)bh * D + d] = __float2bfloat16_rn(0.f);
    if (d == 0 && p.lse != nullptr) p.lse[bh] = -INFINITY;
    return;
  }
  const float* ml = p.part_ml + (size_t)bh * p.nsplit * 2;
  float mx = -INFINITY;
  for (int i = d; i < n; i += D) mx = fmaxf(mx, ml[2 * i]);
  mx = block_reduce(mx, true, red);
  float lsum = 0.f;
  for (int i = d; i < n; i += D) {
    const float e = ex2_approx(ml[2 * i] - mx);
    wsplit[i] = e;
    lsum = fmaf(e, ml[2 * i + 1], lsum);
  }
  lsum = block_reduce(lsum, false, red);  // its barriers also publish wsplit
  const float* po = p.part_o + (size_t)bh * p.nsplit * D + d;
  float acc = 0.f;
  for (int i = 0; i < n; ++i) acc = fmaf(wsplit[i], po[(size_t)i * D], acc);
  const float val = acc / lsum;
  if (p.out_f32)
    reinterpret_cast<float*>(p.out)[(size_t)bh * D + d] = val;
  else
    reinterpret_cast<__nv_bfloat16*>(p.out)[(size_t)bh * D + d] = __float2bfloat16_rn(val);
  if (d == 0 && p.lse != nullptr) p.lse[bh] = (mx + log2f(lsum)) * kLn2;
}

template <int D, int GP>
cudaError_t launch_split(const DecodeLaunch& p, int ngroups, int group) {
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
  dim3 grid(p.nsplit, p.Hkv * ngroups, p.B);
  decode_split_kernel<D, GP><<<grid, C::THREADS, C::SMEM, p.stream>>>(p, ngroups, group);
  return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_gp(const DecodeLaunch& p) {
  const int group = p.Hq / p.Hkv;
  const int gp = decode_heads_per_cta(group);
  const int ngroups = group / gp;
  switch (gp) {
    case 8: return launch_split<D, 8>(p, ngroups, group);
    case 4: return launch_split<D, 4>(p, ngroups, group);
    case 2: return launch_split<D, 2>(p, ngroups, group);
    default: return launch_split<D, 1>(p, ngroups, group);
  }
}

}  // namespace

int decode_stage_keys(int D) { return D == 64 ? DecodeCfg<64, 1>::SK : DecodeCfg<128, 1>::SK; }

int decode_heads_per_cta(int group) {
  for (int gp = 8; gp > 1; gp >>= 1)
    if (group % gp == 0) return gp;
  return 1;
}

cudaError_t launch_decode(const DecodeLaunch& p) {
  cudaError_t e = (p.D == 64) ? dispatch_gp<64>(p) : dispatch_gp<128>(p);
  if (e != cudaSuccess) return e;
  decode_combine_kernel<<<p.B * p.Hq, p.D, p.nsplit * sizeof(float), p.stream>>>(p);
  return cudaGetLastError();
}

}  // namespace attn
