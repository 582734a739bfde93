"""Thin ctypes binding of the C ABI in ``include/attn.h`` (argument marshalling only).

Every function here has the name of the C entry point it calls.  Tensors are
torch tensors on a CUDA device; the binding checks dtypes, shapes and
contiguity, allocates outputs the caller did not pass (torch supplies device
memory), and hands raw pointers plus the current torch stream to the library.
All computation happens in the library's CUDA kernels.  If the library has not
been built, the first call raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn_gb300.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_ALIGNMENT = 3
ATTN_ERR_CUDA = 4
ATTN_ERR_DEVICE_TIMEOUT = 5
ATTN_ERR_DEVICE_BOUNDS = 6
ATTN_ERR_SCRATCH_TOO_SMALL = 7
ATTN_DTYPE_BF16 = 0
ATTN_DTYPE_F32 = 1

# Every symbol include/attn.h declares.
EXPORTED = (
    "attn_fwd",
    "attn_fwd_ex",
    "attn_decode",
    "attn_decode_ex",
    "attn_decode_noalloc",
    "attn_decode_paged",
    "attn_decode_multi",
    "attn_decode_workspace_bytes",
    "attn_get_device_status",
    "attn_status_string",
    "attn_release_workspace",
    "attn_selftest_wait_timeout",
    "attn_version",
)


ATTN_ROPE_NONE = 0
ATTN_ROPE_HALF = 1
ATTN_ROPE_INTERLEAVED = 2
_ROPE_STYLES = {"half": ATTN_ROPE_HALF, "interleaved": ATTN_ROPE_INTERLEAVED}


class attn_rope(ctypes.Structure):
    _fields_ = [("cos", ctypes.c_void_p), ("sin", ctypes.c_void_p), ("max_pos", ctypes.c_int), ("style", ctypes.c_int),
                ("k_out", ctypes.c_void_p)]


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class attn_fwd_params(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
        ("Lq", ctypes.c_int), ("Lkv", ctypes.c_int), ("D", ctypes.c_int),
        ("scale", ctypes.c_float), ("causal", ctypes.c_int), ("out_dtype", ctypes.c_int),
        ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p),
        ("total_q", ctypes.c_int), ("total_k", ctypes.c_int),
        ("stream", ctypes.c_void_p),
        ("rope", attn_rope),
    ]


class attn_decode_paged_params(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("kpages", ctypes.c_void_p), ("vpages", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p), ("kv_lens", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("lse", ctypes.c_void_p),
        ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
        ("page_size", ctypes.c_int), ("max_pages", ctypes.c_int), ("num_pages", ctypes.c_int),
        ("scale", ctypes.c_float), ("out_dtype", ctypes.c_int), ("chunk", ctypes.c_int),
        ("stream", ctypes.c_void_p),
        ("rope", attn_rope),
    ]


class attn_decode_multi_params(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("kcache", ctypes.c_void_p), ("vcache", ctypes.c_void_p),
        ("kv_lens", ctypes.c_void_p), ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("Lq", ctypes.c_int),
        ("Lmax", ctypes.c_int), ("D", ctypes.c_int),
        ("scale", ctypes.c_float), ("out_dtype", ctypes.c_int),
        ("stream", ctypes.c_void_p),
        ("rope", attn_rope),
    ]


class attn_decode_params(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("kcache", ctypes.c_void_p), ("vcache", ctypes.c_void_p),
        ("kv_lens", ctypes.c_void_p), ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
        ("Lmax", ctypes.c_int), ("D", ctypes.c_int),
        ("scale", ctypes.c_float), ("out_dtype", ctypes.c_int), ("chunk", ctypes.c_int),
        ("stream", ctypes.c_void_p),
        ("rope", attn_rope),
    ]


_lib = None
_lock = threading.Lock()


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library once (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"attention library not built: {path} is missing (run __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, I, P]
        lib.attn_fwd.restype = I
        lib.attn_fwd_ex.argtypes = [ctypes.POINTER(attn_fwd_params)]
        lib.attn_fwd_ex.restype = I
        lib.attn_decode.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, P]
        lib.attn_decode.restype = I
        lib.attn_decode_ex.argtypes = [ctypes.POINTER(attn_decode_params)]
        lib.attn_decode_ex.restype = I
        lib.attn_decode_noalloc.argtypes = [ctypes.POINTER(attn_decode_params)]
        lib.attn_decode_noalloc.restype = I
        lib.attn_decode_paged.argtypes = [ctypes.POINTER(attn_decode_paged_params)]
        lib.attn_decode_paged.restype = I
        lib.attn_decode_multi.argtypes = [ctypes.POINTER(attn_decode_multi_params)]
        lib.attn_decode_multi.restype = I
        lib.attn_decode_workspace_bytes.argtypes = [I, I, I, I, I, I]
        lib.attn_decode_workspace_bytes.restype = ctypes.c_ulonglong
        lib.attn_get_device_status.argtypes = [P]
        lib.attn_get_device_status.restype = I
        lib.attn_status_string.argtypes = [I]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_release_workspace.argtypes = []
        lib.attn_release_workspace.restype = None
        lib.attn_selftest_wait_timeout.argtypes = [ctypes.c_uint, P]
        lib.attn_selftest_wait_timeout.restype = I
        lib.attn_version.argtypes = []
        lib.attn_version.restype = I
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != ATTN_OK:
        raise AttnError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype, ndim, shape=None, device=None):
    """Check a tensor argument; ``shape`` and ``device``, when given, must match exactly (outputs are written
    by the kernels over their full extent, so a smaller buffer must never reach the library)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _set_rope(p, rope, D, device, k_shape=None):
    """rope = (cos, sin, style) or (cos, sin, style, k_out): fp32 device tables [max_pos, D/2], "half" or
    "interleaved", and for prefill an optional bf16 tensor shaped like k receiving the rotated keys (None: off)."""
    if rope is None:
        return
    cos, sin, style = rope[:3]
    k_out = rope[3] if len(rope) > 3 else None
    if k_out is not None:
        if k_shape is None:
            raise ValueError("rope k_out is taken by prefill calls only")
        _need(k_out, "rope k_out", torch.bfloat16, len(k_shape), k_shape, device)
        p.rope.k_out = _ptr(k_out)
    for t, name in ((cos, "rope cos"), (sin, "rope sin")):
        _need(t, name, torch.float32, 2)
        if t.device != device or t.shape[1] != D // 2:
            raise ValueError(f"{name} must be [max_pos, D/2] on {device}")
    if cos.shape != sin.shape:
        raise ValueError("rope cos and sin tables differ in shape")
    if style not in _ROPE_STYLES:
        raise ValueError("rope style must be 'half' or 'interleaved'")
    p.rope.cos, p.rope.sin = _ptr(cos), _ptr(sin)
    p.rope.max_pos = cos.shape[0]
    p.rope.style = _ROPE_STYLES[style]


def attn_fwd(q, k, v, out=None, lse=None, causal=True, scale=None, out_dtype=torch.bfloat16,
             want_lse=True, stream=None, rope=None):
    """Dense prefill: q [B,Hq,Lq,D], k/v [B,Hkv,Lkv,D] bf16 -> (out [B,Hq,Lq,D], lse [B,Hq,Lq] fp32).

    ``rope = (cos, sin, style)`` rotates q and k inside the call (fp32 device tables [max_pos, D/2];
    style "half" or "interleaved"); every call of this module takes the same argument."""
    _need(q, "q", torch.bfloat16, 4)
    _need(k, "k", torch.bfloat16, 4, device=q.device)
    _need(v, "v", torch.bfloat16, 4, device=q.device)
    B, Hq, Lq, D = q.shape
    Hkv, Lkv = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Hkv, Lkv, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"k/v shapes {tuple(k.shape)} {tuple(v.shape)} do not match q {tuple(q.shape)}")
    if out is None:
        out = torch.empty((B, Hq, Lq, D), dtype=out_dtype, device=q.device)
    _need(out, "out", out_dtype, 4, (B, Hq, Lq, D), q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 3, (B, Hq, Lq), q.device)
    p = attn_fwd_params()
    p.q, p.k, p.v, p.out, p.lse = (_ptr(t) for t in (q, k, v, out, lse))
    p.B, p.Hq, p.Hkv, p.Lq, p.Lkv, p.D = B, Hq, Hkv, Lq, Lkv, D
    p.scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    p.causal = int(bool(causal))
    p.out_dtype = ATTN_DTYPE_F32 if out_dtype == torch.float32 else ATTN_DTYPE_BF16
    p.stream = _stream_handle(stream, q.device)
    _set_rope(p, rope, D, q.device, tuple(k.shape))
    _check(load().attn_fwd_ex(ctypes.byref(p)), "attn_fwd")
    return out, lse


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, out=None, lse=None,
                    causal=True, scale=None, out_dtype=torch.bfloat16, want_lse=True, stream=None, rope=None):
    """Packed prefill: q [total_q,Hq,D], k/v [total_k,Hkv,D] bf16, cu_seqlens int32 [B+1] on the device."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3, device=q.device)
    _need(v, "v", torch.bfloat16, 3, device=q.device)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1, device=q.device)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1, device=q.device)
    total_q, Hq, D = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    B = cu_seqlens_q.shape[0] - 1
    if cu_seqlens_k.shape[0] != B + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    if out is None:
        out = torch.empty((total_q, Hq, D), dtype=out_dtype, device=q.device)
    _need(out, "out", out_dtype, 3, (total_q, Hq, D), q.device)
    if lse is None and want_lse:
        lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2, (total_q, Hq), q.device)
    p = attn_fwd_params()
    p.q, p.k, p.v, p.out, p.lse = (_ptr(t) for t in (q, k, v, out, lse))
    p.B, p.Hq, p.Hkv, p.Lq, p.Lkv, p.D = B, Hq, Hkv, int(max_seqlen_q), int(max_seqlen_k), D
    p.scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    p.causal = int(bool(causal))
    p.out_dtype = ATTN_DTYPE_F32 if out_dtype == torch.float32 else ATTN_DTYPE_BF16
    p.cu_seqlens_q, p.cu_seqlens_k = _ptr(cu_seqlens_q), _ptr(cu_seqlens_k)
    p.total_q, p.total_k = total_q, total_k
    p.stream = _stream_handle(stream, q.device)
    _set_rope(p, rope, D, q.device, tuple(k.shape))
    _check(load().attn_fwd_ex(ctypes.byref(p)), "attn_fwd_ex")
    return out, lse


def attn_decode(q, kcache, vcache, kv_lens, out=None, lse=None, scale=None, chunk=0,
                out_dtype=torch.bfloat16, want_lse=True, stream=None, rope=None):
    """Decode: q [B,Hq,D], caches [B,Hkv,Lmax,D] bf16, kv_lens int32 [B] -> (out [B,Hq,D], lse [B,Hq])."""
    _need(q, "q", torch.bfloat16, 3)
    _need(kcache, "kcache", torch.bfloat16, 4, device=q.device)
    _need(vcache, "vcache", torch.bfloat16, 4, device=q.device)
    _need(kv_lens, "kv_lens", torch.int32, 1, device=q.device)
    B, Hq, D = q.shape
    Hkv, Lmax = kcache.shape[1], kcache.shape[2]
    if tuple(kcache.shape) != (B, Hkv, Lmax, D) or tuple(vcache.shape) != tuple(kcache.shape):
        raise ValueError("cache shapes do not match q")
    if kv_lens.shape[0] != B:
        raise ValueError("kv_lens must have B entries")
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    _need(out, "out", out_dtype, 3, (B, Hq, D), q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2, (B, Hq), q.device)
    p = attn_decode_params()
    p.q, p.kcache, p.vcache, p.kv_lens, p.out, p.lse = (_ptr(t) for t in (q, kcache, vcache, kv_lens, out, lse))
    p.B, p.Hq, p.Hkv, p.Lmax, p.D = B, Hq, Hkv, Lmax, D
    p.scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    p.out_dtype = ATTN_DTYPE_F32 if out_dtype == torch.float32 else ATTN_DTYPE_BF16
    p.chunk = int(chunk)
    p.stream = _stream_handle(stream, q.device)
    _set_rope(p, rope, D, q.device)
    _check(load().attn_decode_ex(ctypes.byref(p)), "attn_decode")
    return out, lse


def attn_decode_paged(q, kpages, vpages, block_table, kv_lens, out=None, lse=None, scale=None, chunk=0,
                      out_dtype=torch.bfloat16, want_lse=True, stream=None, rope=None):
    """Decode over a paged cache: pages [num_pages,Hkv,page_size,D] bf16, block_table int32 [B,max_pages]."""
    _need(q, "q", torch.bfloat16, 3)
    _need(kpages, "kpages", torch.bfloat16, 4, device=q.device)
    _need(vpages, "vpages", torch.bfloat16, 4, device=q.device)
    _need(block_table, "block_table", torch.int32, 2, device=q.device)
    _need(kv_lens, "kv_lens", torch.int32, 1, device=q.device)
    B, Hq, D = q.shape
    num_pages, Hkv, page_size = kpages.shape[0], kpages.shape[1], kpages.shape[2]
    if tuple(kpages.shape) != (num_pages, Hkv, page_size, D) or tuple(vpages.shape) != tuple(kpages.shape):
        raise ValueError("page pool shapes do not match q")
    if block_table.shape[0] != B or kv_lens.shape[0] != B:
        raise ValueError("block_table and kv_lens must have B rows")
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    _need(out, "out", out_dtype, 3, (B, Hq, D), q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2, (B, Hq), q.device)
    p = attn_decode_paged_params()
    p.q, p.kpages, p.vpages = _ptr(q), _ptr(kpages), _ptr(vpages)
    p.block_table, p.kv_lens, p.out, p.lse = _ptr(block_table), _ptr(kv_lens), _ptr(out), _ptr(lse)
    p.B, p.Hq, p.Hkv, p.D = B, Hq, Hkv, D
    p.page_size, p.max_pages, p.num_pages = page_size, block_table.shape[1], num_pages
    p.scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    p.out_dtype = ATTN_DTYPE_F32 if out_dtype == torch.float32 else ATTN_DTYPE_BF16
    p.chunk = int(chunk)
    p.stream = _stream_handle(stream, q.device)
    _set_rope(p, rope, D, q.device)
    _check(load().attn_decode_paged(ctypes.byref(p)), "attn_decode_paged")
    return out, lse


def attn_decode_multi(q, kcache, vcache, kv_lens, out=None, lse=None, scale=None, out_dtype=torch.bfloat16,
                      want_lse=True, stream=None, rope=None):
    """Multi-token decode: q [B,Hq,Lq,D], caches [B,Hkv,Lmax,D] bf16, kv_lens int32 [B] counting the new tokens'
    own keys -> (out [B,Hq,Lq,D], lse [B,Hq,Lq])."""
    _need(q, "q", torch.bfloat16, 4)
    _need(kcache, "kcache", torch.bfloat16, 4, device=q.device)
    _need(vcache, "vcache", torch.bfloat16, 4, device=q.device)
    _need(kv_lens, "kv_lens", torch.int32, 1, device=q.device)
    B, Hq, Lq, D = q.shape
    Hkv, Lmax = kcache.shape[1], kcache.shape[2]
    if tuple(kcache.shape) != (B, Hkv, Lmax, D) or tuple(vcache.shape) != tuple(kcache.shape):
        raise ValueError("cache shapes do not match q")
    if kv_lens.shape[0] != B:
        raise ValueError("kv_lens must have B entries")
    if out is None:
        out = torch.empty((B, Hq, Lq, D), dtype=out_dtype, device=q.device)
    _need(out, "out", out_dtype, 4, (B, Hq, Lq, D), q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 3, (B, Hq, Lq), q.device)
    p = attn_decode_multi_params()
    p.q, p.kcache, p.vcache, p.kv_lens, p.out, p.lse = (_ptr(t) for t in (q, kcache, vcache, kv_lens, out, lse))
    p.B, p.Hq, p.Hkv, p.Lq, p.Lmax, p.D = B, Hq, Hkv, Lq, Lmax, D
    p.scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    p.out_dtype = ATTN_DTYPE_F32 if out_dtype == torch.float32 else ATTN_DTYPE_BF16
    p.stream = _stream_handle(stream, q.device)
    _set_rope(p, rope, D, q.device)
    _check(load().attn_decode_multi(ctypes.byref(p)), "attn_decode_multi")
    return out, lse


def attn_decode_noalloc(q, kcache, vcache, kv_lens, out, lse=None, scale=None, chunk=0, stream=None, rope=None):
    """Decode through the entry point that allocates no device memory.

    For callers that cannot allocate (inside CUDA graph capture, engines that
    hand all of HBM to their own pool, latency paths that cannot take
    cudaMalloc's synchronisation).  ``out`` (and ``lse`` if wanted) must be
    passed in; the split-KV partials go to a fixed 4 MiB buffer inside the
    library, shared by every call on the device, so calls that may overlap on
    the GPU must be ordered on one stream.  The first call on a device does a
    one-time address lookup and should not be inside a stream capture.
    """
    _need(q, "q", torch.bfloat16, 3)
    _need(kcache, "kcache", torch.bfloat16, 4, device=q.device)
    _need(vcache, "vcache", torch.bfloat16, 4, device=q.device)
    _need(kv_lens, "kv_lens", torch.int32, 1, device=q.device)
    B, Hq, D = q.shape
    Hkv, Lmax = kcache.shape[1], kcache.shape[2]
    if tuple(kcache.shape) != (B, Hkv, Lmax, D) or tuple(vcache.shape) != tuple(kcache.shape):
        raise ValueError("cache shapes do not match q")
    if kv_lens.shape[0] != B:
        raise ValueError("kv_lens must have B entries")
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out must be bf16 or fp32")
    _need(out, "out", out.dtype, 3, (B, Hq, D), q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2, (B, Hq), q.device)
    p = attn_decode_params()
    p.q, p.kcache, p.vcache, p.kv_lens, p.out, p.lse = (_ptr(t) for t in (q, kcache, vcache, kv_lens, out, lse))
    p.B, p.Hq, p.Hkv, p.Lmax, p.D = B, Hq, Hkv, Lmax, D
    p.scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    p.out_dtype = ATTN_DTYPE_F32 if out.dtype == torch.float32 else ATTN_DTYPE_BF16
    p.chunk = int(chunk)
    p.stream = _stream_handle(stream, q.device)
    _set_rope(p, rope, D, q.device)
    _check(load().attn_decode_noalloc(ctypes.byref(p)), "attn_decode_noalloc")
    return out, lse


def attn_decode_workspace_bytes(B, Hq, Hkv, Lmax, D, chunk=0) -> int:
    return int(load().attn_decode_workspace_bytes(B, Hq, Hkv, Lmax, D, chunk))


def attn_get_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    h = None if stream is None else ctypes.c_void_p(stream.cuda_stream)
    return int(load().attn_get_device_status(h))


def attn_release_workspace():
    load().attn_release_workspace()


def attn_version() -> int:
    return int(load().attn_version())


def attn_selftest_wait_timeout(limit_us=1000, stream=None):
    """Run the bounded-wait timeout path on the current device (no fault): afterwards the device status word
    holds ATTN_ERR_DEVICE_TIMEOUT."""
    dev = torch.device("cuda", torch.cuda.current_device())
    _check(load().attn_selftest_wait_timeout(int(limit_us), _stream_handle(stream, dev)), "attn_selftest_wait_timeout")
