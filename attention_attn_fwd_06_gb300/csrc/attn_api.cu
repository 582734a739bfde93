// attn_api.cu -- the C ABI declared in include/attn.h.
//
// Host side only: argument validation (before anything touches the device),
// the sm_103 device check, the per-device split-KV workspace and status word,
// and the kernel launches.  No compute happens here and there is no CPU path.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/attn.h"
#include "kernels.h"

// Device status word: kernels record the first problem they see (a kv_len out
// of range, an expired pipeline wait); attn_get_device_status() reads and
// clears it.  Each device holds its own copy.
__device__ unsigned g_attn_device_status;

namespace {

constexpr int kMaxDevices = 64;
// Decode workspace layout: [counters: kDecodeCounterSlots x u32][part_o][part_ml].
// The counter area must be zero before the first call; the kernel leaves it zero.
constexpr size_t kCounterBytes = size_t(attn::kDecodeCounterSlots) * sizeof(unsigned);

struct DeviceState {
  bool probed = false;
  int support = ATTN_OK;  // ATTN_ERR_UNSUPPORTED when the device is not sm_103
  int num_sms = 0;
  unsigned* status = nullptr;
  void* ws = nullptr;
  size_t ws_bytes = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Fixed split-KV scratch for attn_decode_noalloc: 4 MiB of fp32 partials per
// device, part of the library's device image (no runtime allocation).
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;
__device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];
// Device address of g_noalloc_scratch per device (host code cannot use the
// symbol itself as a pointer), looked up on the first no-alloc call there.
float* g_noalloc_ptr[kMaxDevices] = {};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ATTN_FAULT_INJECT=skip_arrive (read at each decode and prefill call): CTA 0 of the kernel withholds one
// arrival -- decode a pipeline-slot release, prefill and multi-token decode a P-ready signal -- so a bounded
// wait runs out and ATTN_ERR_DEVICE_TIMEOUT is recorded: a test of the failure path on a real kernel that
// neither faults nor hangs the GPU.
int fault_skip_arrive() {
  const char* v = std::getenv("ATTN_FAULT_INJECT");
  return (v != nullptr && std::strcmp(v, "skip_arrive") == 0) ? 1 : 0;
}
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Looks up (and on first use probes) the current device.  Caller holds g_mu.
int device_state_locked(DeviceState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return ATTN_ERR_UNSUPPORTED;
  }
  DeviceState& s = g_dev[dev];
  if (!s.probed) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    s.support = (major == 10 && minor == 3) ? ATTN_OK : ATTN_ERR_UNSUPPORTED;
    s.num_sms = sms;
    if (s.support == ATTN_OK) {
      if (cudaGetSymbolAddress(reinterpret_cast<void**>(&s.status), g_attn_device_status) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
      }
    }
    s.probed = true;
  }
  *out = &s;
  return s.support;
}

int map_cuda(cudaError_t e) {
  if (e == cudaSuccess) return ATTN_OK;
  if (e == cudaErrorNotSupported) return ATTN_ERR_UNSUPPORTED;
  return ATTN_ERR_CUDA;
}

// Ensures the workspace of `s` holds `bytes`.  Refuses to allocate while the
// stream is being captured into a CUDA graph.  Caller holds g_mu.
int ensure_workspace_locked(DeviceState& s, size_t bytes, cudaStream_t stream) {
  if (bytes <= s.ws_bytes) return ATTN_OK;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  if (cap != cudaStreamCaptureStatusNone) return ATTN_ERR_INVALID_ARG;
  if (s.ws != nullptr) {
    cudaFree(s.ws);  // synchronises the device: no earlier decode can still be using it
    s.ws = nullptr;
    s.ws_bytes = 0;
  }
  if (cudaMalloc(&s.ws, bytes) != cudaSuccess) {
    cudaGetLastError();
    s.ws = nullptr;
    return ATTN_ERR_CUDA;
  }
  if (cudaMemset(s.ws, 0, kCounterBytes) != cudaSuccess) {  // counters start at zero
    cudaGetLastError();
    cudaFree(s.ws);
    s.ws = nullptr;
    return ATTN_ERR_CUDA;
  }
  s.ws_bytes = bytes;
  return ATTN_OK;
}

struct DecodeShape {
  int grid = 0;               // CTAs of the persistent launch
  size_t part_o_elems = 0;    // 2 * grid * GP * D
  size_t part_ml_elems = 0;   // 2 * grid * GP * 2
  size_t bytes = 0;           // counters + partials
};

// The stream-K split gives every CTA an equal slice of the key space and each
// CTA at most two partial rows, so the partial area depends on the grid, the
// heads per CTA and D -- not on the batch or the cache length.
DecodeShape decode_shape(int Hq, int Hkv, int D, int num_sms) {
  DecodeShape s;
  const int gp = attn::decode_heads_per_cta(Hq / Hkv);
  s.grid = attn::decode_grid(num_sms, Hq / Hkv);
  s.part_o_elems = (size_t)2 * s.grid * gp * D;
  s.part_ml_elems = (size_t)2 * s.grid * gp * 2;
  s.bytes = kCounterBytes + (s.part_o_elems + s.part_ml_elems) * sizeof(float);
  return s;
}

// Rows of per-row counters the decode kernel uses for these sizes.
long long decode_counter_rows(int B, int Hq, int Hkv) {
  const int group = Hq / Hkv;
  return (long long)B * Hkv * (group / attn::decode_heads_per_cta(group));
}

int validate_decode(const attn_decode_params* p) {
  if (p == nullptr) return ATTN_ERR_INVALID_ARG;
  if (p->B < 0 || p->Hq <= 0 || p->Hkv <= 0 || p->Lmax < 0 || p->D <= 0) return ATTN_ERR_INVALID_ARG;
  if (p->Hq % p->Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (p->D != 64 && p->D != 128) return ATTN_ERR_UNSUPPORTED;
  if (p->out_dtype != ATTN_DTYPE_BF16 && p->out_dtype != ATTN_DTYPE_F32) return ATTN_ERR_INVALID_ARG;
  if (p->chunk < 0 || p->chunk > (1 << 20)) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(p->scale)) return ATTN_ERR_INVALID_ARG;  // NaN or infinite scale
  if (p->B == 0) return ATTN_OK;
  if (p->q == nullptr || p->kcache == nullptr || p->vcache == nullptr || p->kv_lens == nullptr ||
      p->out == nullptr)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(p->q) || !aligned16(p->kcache) || !aligned16(p->vcache) || !aligned16(p->out) ||
      !aligned4(p->kv_lens) || (p->lse != nullptr && !aligned4(p->lse)))
    return ATTN_ERR_ALIGNMENT;
  if (p->B > 65535 || p->Hkv > 65535 || (long long)p->B * p->Hq > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

int validate_fwd(const attn_fwd_params* p) {
  if (p == nullptr) return ATTN_ERR_INVALID_ARG;
  if (p->B < 0 || p->Hq <= 0 || p->Hkv <= 0 || p->Lq < 0 || p->Lkv < 0 || p->D <= 0)
    return ATTN_ERR_INVALID_ARG;
  if (p->Hq % p->Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (p->D != 64 && p->D != 128) return ATTN_ERR_UNSUPPORTED;
  if (p->causal != 0 && p->causal != 1) return ATTN_ERR_INVALID_ARG;
  if (p->out_dtype != ATTN_DTYPE_BF16 && p->out_dtype != ATTN_DTYPE_F32) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(p->scale)) return ATTN_ERR_INVALID_ARG;  // NaN or infinite scale
  const bool varlen = p->cu_seqlens_q != nullptr || p->cu_seqlens_k != nullptr;
  if (varlen) {
    if (p->cu_seqlens_q == nullptr || p->cu_seqlens_k == nullptr) return ATTN_ERR_INVALID_ARG;
    if (p->total_q < 0 || p->total_k < 0) return ATTN_ERR_INVALID_ARG;
    if (!aligned4(p->cu_seqlens_q) || !aligned4(p->cu_seqlens_k)) return ATTN_ERR_ALIGNMENT;
  }
  if (p->B == 0 || p->Lq == 0 || (varlen && p->total_q == 0)) return ATTN_OK;
  const bool no_keys = varlen ? p->total_k == 0 : p->Lkv == 0;  // then k and v are never read
  if (p->q == nullptr || p->out == nullptr || (!no_keys && (p->k == nullptr || p->v == nullptr)))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(p->q) || !aligned16(p->k) || !aligned16(p->v) || !aligned16(p->out) ||
      (p->lse != nullptr && !aligned4(p->lse)))
    return ATTN_ERR_ALIGNMENT;
  if (p->B > 65535 || (long long)p->B * p->Hq > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

// Checks a rotary-embedding argument whose largest position is max_needed - 1 (0: nothing rotated).
int validate_rope(const attn_rope& r, int D, long long max_needed) {
  if (r.style == ATTN_ROPE_NONE || r.cos == nullptr) return ATTN_OK;
  if (r.style != ATTN_ROPE_HALF && r.style != ATTN_ROPE_INTERLEAVED) return ATTN_ERR_INVALID_ARG;
  if (r.sin == nullptr || r.max_pos <= 0) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(r.cos) || !aligned16(r.sin)) return ATTN_ERR_ALIGNMENT;
  if (max_needed > r.max_pos) return ATTN_ERR_INVALID_ARG;
  if ((long long)r.max_pos * (D / 2) > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

attn::RopeArgs rope_args(const attn_rope& r) {
  attn::RopeArgs a{};
  if (r.style != ATTN_ROPE_NONE && r.cos != nullptr) {
    a.cos = r.cos;
    a.sin = r.sin;
    a.max_pos = r.max_pos;
    a.style = r.style;
  }
  return a;
}

bool is_empty_fwd(const attn_fwd_params* p) {
  const bool varlen = p->cu_seqlens_q != nullptr;
  return p->B == 0 || p->Lq == 0 || (varlen && p->total_q == 0);
}

}  // namespace

extern "C" {

int attn_version(void) { return 100; }

int attn_selftest_wait_timeout(unsigned int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return ATTN_ERR_INVALID_ARG;
  DeviceState* s = nullptr;
  int st;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    st = device_state_locked(&s);
  }
  if (st != ATTN_OK) return st;
  return map_cuda(attn::launch_selftest_timeout((unsigned long long)limit_us * 1000ull, s->status,
                                                static_cast<cudaStream_t>(stream)));
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_ALIGNMENT: return "ATTN_ERR_ALIGNMENT";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_DEVICE_TIMEOUT: return "ATTN_ERR_DEVICE_TIMEOUT";
    case ATTN_ERR_DEVICE_BOUNDS: return "ATTN_ERR_DEVICE_BOUNDS";
    case ATTN_ERR_SCRATCH_TOO_SMALL: return "ATTN_ERR_SCRATCH_TOO_SMALL";
    default: return "ATTN_STATUS_UNKNOWN";
  }
}

unsigned long long attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Lmax, int D, int chunk) {
  attn_decode_params p = {};
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Lmax = Lmax; p.D = D; p.chunk = chunk;
  p.q = p.kcache = p.vcache = reinterpret_cast<const void*>(16);
  p.kv_lens = reinterpret_cast<const int*>(16);
  p.out = reinterpret_cast<void*>(16);
  if (validate_decode(&p) != ATTN_OK || B == 0) return 0;
  if (2 + decode_counter_rows(B, Hq, Hkv) > attn::kDecodeCounterSlots) return 0;
  int sms = 0;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* s = nullptr;
    if (device_state_locked(&s) == ATTN_OK) sms = s->num_sms;
  }
  return decode_shape(Hq, Hkv, D, sms).bytes;
}

int attn_decode_ex(const attn_decode_params* p) {
  int st = validate_decode(p);
  if (st != ATTN_OK) return st;
  st = validate_rope(p->rope, p->D, p->Lmax);
  if (st != ATTN_OK) return st;
  if (p->B == 0) return ATTN_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(p->stream);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  st = device_state_locked(&s);
  if (st != ATTN_OK) return st;
  if (2 + decode_counter_rows(p->B, p->Hq, p->Hkv) > attn::kDecodeCounterSlots) return ATTN_ERR_UNSUPPORTED;
  const DecodeShape sh = decode_shape(p->Hq, p->Hkv, p->D, s->num_sms);
  st = ensure_workspace_locked(*s, sh.bytes, stream);
  if (st != ATTN_OK) return st;
  attn::DecodeLaunch L{};
  L.q = p->q;
  L.kcache = p->kcache;
  L.vcache = p->vcache;
  L.kv_lens = p->kv_lens;
  L.out = p->out;
  L.lse = p->lse;
  L.counters = static_cast<unsigned*>(s->ws);
  L.part_o = reinterpret_cast<float*>(static_cast<char*>(s->ws) + kCounterBytes);
  L.part_ml = L.part_o + sh.part_o_elems;
  L.B = p->B;
  L.Hq = p->Hq;
  L.Hkv = p->Hkv;
  L.Lmax = p->Lmax;
  L.D = p->D;
  L.min_keys = p->chunk > 0 ? p->chunk : 64;
  L.scale = p->scale;
  L.out_f32 = p->out_dtype == ATTN_DTYPE_F32;
  L.status = s->status;
  L.fault_skip_arrive = fault_skip_arrive();
  L.rope = rope_args(p->rope);
  L.stream = stream;
  return map_cuda(attn::launch_decode(L, s->num_sms));
}

int attn_decode_noalloc(const attn_decode_params* p) {
  int st = validate_decode(p);
  if (st != ATTN_OK) return st;
  st = validate_rope(p->rope, p->D, p->Lmax);
  if (st != ATTN_OK) return st;
  if (p->B == 0) return ATTN_OK;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  st = device_state_locked(&s);
  if (st != ATTN_OK) return st;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  if (g_noalloc_ptr[dev] == nullptr) {
    // One-time set-up on this device (it is current).  Its memset and synchronise would invalidate a stream
    // capture in progress, so a first call made inside one is refused before anything touches the device.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(static_cast<cudaStream_t>(p->stream), &cap) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    if (cap != cudaStreamCaptureStatusNone) return ATTN_ERR_INVALID_ARG;
    // Resolve the scratch array's device address.
    float* ptr = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    // Its counter area must start at zero; the kernel keeps it zero afterwards.
    if (cudaMemset(ptr, 0, kCounterBytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = ptr;
  }
  const DecodeShape sh = decode_shape(p->Hq, p->Hkv, p->D, s->num_sms);
  if (2 + decode_counter_rows(p->B, p->Hq, p->Hkv) > attn::kDecodeCounterSlots || sh.bytes > kNoAllocScratchBytes)
    return ATTN_ERR_SCRATCH_TOO_SMALL;
  attn::DecodeLaunch L{};
  L.q = p->q;
  L.kcache = p->kcache;
  L.vcache = p->vcache;
  L.kv_lens = p->kv_lens;
  L.out = p->out;
  L.lse = p->lse;
  L.counters = reinterpret_cast<unsigned*>(g_noalloc_ptr[dev]);
  L.part_o = g_noalloc_ptr[dev] + kCounterBytes / sizeof(float);
  L.part_ml = L.part_o + sh.part_o_elems;
  L.B = p->B;
  L.Hq = p->Hq;
  L.Hkv = p->Hkv;
  L.Lmax = p->Lmax;
  L.D = p->D;
  L.min_keys = p->chunk > 0 ? p->chunk : 64;
  L.scale = p->scale;
  L.out_f32 = p->out_dtype == ATTN_DTYPE_F32;
  L.status = s->status;
  L.fault_skip_arrive = fault_skip_arrive();
  L.rope = rope_args(p->rope);
  L.stream = static_cast<cudaStream_t>(p->stream);
  return map_cuda(attn::launch_decode(L, s->num_sms));
}

int attn_decode_paged(const attn_decode_paged_params* pp) {
  if (pp == nullptr) return ATTN_ERR_INVALID_ARG;
  if (pp->page_size < 8 || pp->page_size > 65536 || pp->max_pages < 1 || pp->num_pages < 1)
    return ATTN_ERR_INVALID_ARG;
  const long long lmax = (long long)pp->max_pages * pp->page_size;
  if (lmax > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  // Validate everything else as the contiguous call does (same meaning of every other field).
  attn_decode_params p = {};
  p.q = pp->q;
  p.kcache = pp->kpages;
  p.vcache = pp->vpages;
  p.kv_lens = pp->kv_lens;
  p.out = pp->out;
  p.lse = pp->lse;
  p.B = pp->B;
  p.Hq = pp->Hq;
  p.Hkv = pp->Hkv;
  p.Lmax = (int)lmax;
  p.D = pp->D;
  p.scale = pp->scale;
  p.out_dtype = pp->out_dtype;
  p.chunk = pp->chunk;
  p.stream = pp->stream;
  p.rope = pp->rope;
  int st = validate_decode(&p);
  if (st != ATTN_OK) return st;
  st = validate_rope(p.rope, p.D, p.Lmax);
  if (st != ATTN_OK) return st;
  if (p.B == 0) return ATTN_OK;
  if (pp->block_table == nullptr) return ATTN_ERR_INVALID_ARG;
  if (!aligned4(pp->block_table)) return ATTN_ERR_ALIGNMENT;
  cudaStream_t stream = static_cast<cudaStream_t>(p.stream);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  st = device_state_locked(&s);
  if (st != ATTN_OK) return st;
  if (2 + decode_counter_rows(p.B, p.Hq, p.Hkv) > attn::kDecodeCounterSlots) return ATTN_ERR_UNSUPPORTED;
  const DecodeShape sh = decode_shape(p.Hq, p.Hkv, p.D, s->num_sms);
  st = ensure_workspace_locked(*s, sh.bytes, stream);
  if (st != ATTN_OK) return st;
  attn::DecodeLaunch L{};
  L.q = p.q;
  L.kcache = p.kcache;
  L.vcache = p.vcache;
  L.block_table = pp->block_table;
  L.page_size = pp->page_size;
  L.max_pages = pp->max_pages;
  L.num_pages = pp->num_pages;
  L.kv_lens = p.kv_lens;
  L.out = p.out;
  L.lse = p.lse;
  L.counters = static_cast<unsigned*>(s->ws);
  L.part_o = reinterpret_cast<float*>(static_cast<char*>(s->ws) + kCounterBytes);
  L.part_ml = L.part_o + sh.part_o_elems;
  L.B = p.B;
  L.Hq = p.Hq;
  L.Hkv = p.Hkv;
  L.Lmax = p.Lmax;
  L.D = p.D;
  L.min_keys = p.chunk > 0 ? p.chunk : 64;
  L.scale = p.scale;
  L.out_f32 = p.out_dtype == ATTN_DTYPE_F32;
  L.status = s->status;
  L.fault_skip_arrive = fault_skip_arrive();
  L.rope = rope_args(p.rope);
  L.stream = stream;
  return map_cuda(attn::launch_decode(L, s->num_sms));
}

int attn_decode_multi(const attn_decode_multi_params* p) {
  if (p == nullptr) return ATTN_ERR_INVALID_ARG;
  if (p->Lq < 1) return ATTN_ERR_INVALID_ARG;
  // Everything but q/out's token axis means what it means for attn_decode_ex.
  attn_decode_params d = {};
  d.q = p->q;
  d.kcache = p->kcache;
  d.vcache = p->vcache;
  d.kv_lens = p->kv_lens;
  d.out = p->out;
  d.lse = p->lse;
  d.B = p->B;
  d.Hq = p->Hq;
  d.Hkv = p->Hkv;
  d.Lmax = p->Lmax;
  d.D = p->D;
  d.scale = p->scale;
  d.out_dtype = p->out_dtype;
  d.stream = p->stream;
  int st = validate_decode(&d);
  if (st != ATTN_OK) return st;
  st = validate_rope(p->rope, p->D, p->Lmax);
  if (st != ATTN_OK) return st;
  if (p->B == 0) return ATTN_OK;
  const long long rows = (long long)(p->Hq / p->Hkv) * p->Lq;
  if (rows > 128) return ATTN_ERR_UNSUPPORTED;
  if ((long long)p->B * p->Hq * p->Lq > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  if (2 + (long long)p->B * p->Hkv > attn::kDecodeCounterSlots) return ATTN_ERR_UNSUPPORTED;
  cudaStream_t stream = static_cast<cudaStream_t>(p->stream);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  st = device_state_locked(&s);
  if (st != ATTN_OK) return st;
  const size_t slots = (size_t)2 * attn::decode_multi_grid(s->num_sms);
  const size_t part_o_elems = slots * (size_t)rows * p->D;
  const size_t part_ml_elems = slots * (size_t)rows * 2;
  st = ensure_workspace_locked(*s, kCounterBytes + (part_o_elems + part_ml_elems) * sizeof(float), stream);
  if (st != ATTN_OK) return st;
  attn::DecodeMultiLaunch L{};
  L.q = p->q;
  L.kcache = p->kcache;
  L.vcache = p->vcache;
  L.kv_lens = p->kv_lens;
  L.out = p->out;
  L.lse = p->lse;
  L.counters = static_cast<unsigned*>(s->ws);
  L.part_o = reinterpret_cast<float*>(static_cast<char*>(s->ws) + kCounterBytes);
  L.part_ml = L.part_o + part_o_elems;
  L.B = p->B;
  L.Hq = p->Hq;
  L.Hkv = p->Hkv;
  L.Lq = p->Lq;
  L.Lmax = p->Lmax;
  L.D = p->D;
  L.scale = p->scale;
  L.out_f32 = p->out_dtype == ATTN_DTYPE_F32;
  L.num_sms = s->num_sms;
  L.status = s->status;
  L.rope = rope_args(p->rope);
  L.fault_skip_arrive = fault_skip_arrive();
  L.stream = stream;
  return map_cuda(attn::launch_decode_multi(L));
}

int attn_decode(const void* q, const void* kcache, const void* vcache, const int* kv_lens, void* out, float* lse,
                int B, int Hq, int Hkv, int Lmax, int D, float scale, void* stream) {
  attn_decode_params p = {};
  p.q = q;
  p.kcache = kcache;
  p.vcache = vcache;
  p.kv_lens = kv_lens;
  p.out = out;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Lmax = Lmax;
  p.D = D;
  p.scale = scale;
  p.out_dtype = ATTN_DTYPE_BF16;
  p.chunk = 0;
  p.stream = stream;
  return attn_decode_ex(&p);
}

int attn_fwd_ex(const attn_fwd_params* p) {
  int st = validate_fwd(p);
  if (st != ATTN_OK) return st;
  // positions reach Lkv - 1 (keys and the last query); a dense call with Lq > Lkv would place queries before 0
  st = validate_rope(p->rope, p->D, p->Lkv);
  if (st != ATTN_OK) return st;
  const bool rope_on = p->rope.style != ATTN_ROPE_NONE && p->rope.cos != nullptr;
  if (rope_on && p->cu_seqlens_q == nullptr && p->Lq > p->Lkv) return ATTN_ERR_INVALID_ARG;
  if (rope_on && p->rope.k_out != nullptr && !aligned16(p->rope.k_out)) return ATTN_ERR_ALIGNMENT;
  if (is_empty_fwd(p)) return ATTN_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(p->stream);
  DeviceState* s = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    st = device_state_locked(&s);
  }
  if (st != ATTN_OK) return st;
  const void* kk = p->k;
  const bool varlen = p->cu_seqlens_q != nullptr;
  const long long krows = varlen ? (long long)p->total_k * p->Hkv : (long long)p->B * p->Hkv * p->Lkv;
  const void* qq = p->q;
  const long long qrows = varlen ? (long long)p->total_q * p->Hq : (long long)p->B * p->Hq * p->Lq;
  if (rope_on && krows > 0) {
    // rotate the keys once (into k_out or the workspace) and the queries (into the workspace), then attend over
    // the rotated copies
    void* kdst = p->rope.k_out;
    void* qdst = nullptr;
    {
      const size_t kbytes = kdst == nullptr ? (size_t)krows * p->D * 2 : 0;
      std::lock_guard<std::mutex> lock(g_mu);
      st = ensure_workspace_locked(*s, kCounterBytes + kbytes + (size_t)qrows * p->D * 2, stream);
      if (st != ATTN_OK) return st;
      if (kdst == nullptr) kdst = static_cast<char*>(s->ws) + kCounterBytes;
      qdst = static_cast<char*>(s->ws) + kCounterBytes + kbytes;
    }
    attn::RopeRowsLaunch R{};
    R.src = p->k;
    R.dst = kdst;
    R.cu = varlen ? p->cu_seqlens_k : nullptr;
    R.B = p->B;
    R.H = p->Hkv;
    R.L = p->Lkv;
    R.D = p->D;
    R.total = p->total_k;
    R.rope = rope_args(p->rope);
    R.status = s->status;
    R.stream = stream;
    st = map_cuda(attn::launch_rope_rows(R));
    if (st != ATTN_OK) return st;
    kk = kdst;
    attn::RopeRowsLaunch Rq = R;  // query i of a sequence sits at i + Lkv - Lq
    Rq.src = p->q;
    Rq.dst = qdst;
    Rq.cu = varlen ? p->cu_seqlens_q : nullptr;
    Rq.cu_kv = varlen ? p->cu_seqlens_k : nullptr;
    Rq.H = p->Hq;
    Rq.L = p->Lq;
    Rq.total = p->total_q;
    Rq.pos_off = varlen ? 0 : p->Lkv - p->Lq;
    st = map_cuda(attn::launch_rope_rows(Rq));
    if (st != ATTN_OK) return st;
    qq = qdst;
  }
  attn::PrefillLaunch L{};
  L.q = qq;
  L.k = kk;
  L.v = p->v;
  L.out = p->out;
  L.lse = p->lse;
  L.B = p->B;
  L.Hq = p->Hq;
  L.Hkv = p->Hkv;
  L.Lq = p->Lq;
  L.Lkv = p->Lkv;
  L.D = p->D;
  L.scale = p->scale;
  L.causal = p->causal;
  L.out_f32 = p->out_dtype == ATTN_DTYPE_F32;
  L.cu_q = p->cu_seqlens_q;
  L.cu_k = p->cu_seqlens_k;
  L.total_q = p->total_q;
  L.total_k = p->total_k;
  L.num_sms = s->num_sms;
  L.status = s->status;
  L.fault_skip_arrive = fault_skip_arrive();
  L.stream = stream;
  return map_cuda(attn::launch_prefill(L));
}

int attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq, int Hkv, int Lq,
             int Lkv, int D, float scale, int causal, void* stream) {
  attn_fwd_params p = {};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Lq = Lq;
  p.Lkv = Lkv;
  p.D = D;
  p.scale = scale;
  p.causal = causal;
  p.out_dtype = ATTN_DTYPE_BF16;
  p.stream = stream;
  return attn_fwd_ex(&p);
}

int attn_get_device_status(void* stream) {
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  int st = device_state_locked(&s);
  if (st != ATTN_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  unsigned v = 0;
  if (cudaMemcpy(&v, s->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  const unsigned zero = 0;
  if (cudaMemcpy(s->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
  if (v == ATTN_ERR_DEVICE_TIMEOUT) {
    // A decode that gave up part-way may have left its work counters armed: clear them.
    int dev = -1;
    cudaGetDevice(&dev);
    if (s->ws != nullptr) cudaMemset(s->ws, 0, kCounterBytes);
    if (dev >= 0 && dev < kMaxDevices && g_noalloc_ptr[dev] != nullptr) cudaMemset(g_noalloc_ptr[dev], 0, kCounterBytes);
    cudaDeviceSynchronize();
    cudaGetLastError();
  }
  return static_cast<int>(v);
}

void attn_release_workspace(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return;
  }
  DeviceState& s = g_dev[dev];
  if (s.ws != nullptr) cudaFree(s.ws);
  s.ws = nullptr;
  s.ws_bytes = 0;
}

}  // extern "C"
