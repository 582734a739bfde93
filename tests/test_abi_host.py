"""Host-side checks of the C ABI that need no GPU.

The library must build for sm_103a, load on a machine without a GPU, export
every entry point include/attn.h declares, and reject bad arguments with the
documented status codes before touching the device.  A well-formed compute
call on a machine without an sm_103 device must fail (no CPU fallback).
"""
import ctypes
import os
import re

import pytest

from attention_attn_fwd_06_gb300 import binding as B
from attention_attn_fwd_06_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return B.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_ ]+\**\s*\**(attn_[a-z0-9_]+)\s*\(", text, flags=re.M)))


def test_header_declares_expected_entry_points():
    assert declared_functions() == sorted(B.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert B.status_string(B.ATTN_OK) == "ATTN_OK"
    assert B.status_string(B.ATTN_ERR_DEVICE_TIMEOUT) == "ATTN_ERR_DEVICE_TIMEOUT"
    assert B.status_string(99) == "ATTN_STATUS_UNKNOWN"
    assert lib.attn_version() >= 100


FAKE = 1 << 20  # 16-byte aligned, never dereferenced: validation happens first


def fwd(lib, **kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, lse=None, B=1, Hq=4, Hkv=2, Lq=8, Lkv=8, D=128,
                scale=0.1, causal=1, stream=None)
    args.update(kw)
    return lib.attn_fwd(args["q"], args["k"], args["v"], args["out"], args["lse"], args["B"], args["Hq"],
                        args["Hkv"], args["Lq"], args["Lkv"], args["D"], ctypes.c_float(args["scale"]),
                        args["causal"], args["stream"])


def dec(lib, **kw):
    args = dict(q=FAKE, kc=FAKE, vc=FAKE, lens=FAKE, out=FAKE, lse=None, B=2, Hq=8, Hkv=2, Lmax=64, D=128,
                scale=0.1, stream=None)
    args.update(kw)
    return lib.attn_decode(args["q"], args["kc"], args["vc"], args["lens"], args["out"], args["lse"], args["B"],
                           args["Hq"], args["Hkv"], args["Lmax"], args["D"], ctypes.c_float(args["scale"]),
                           args["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), B.ATTN_ERR_INVALID_ARG),
    (dict(out=None), B.ATTN_ERR_INVALID_ARG),
    (dict(Hq=3, Hkv=2), B.ATTN_ERR_INVALID_ARG),
    (dict(Hkv=0), B.ATTN_ERR_INVALID_ARG),
    (dict(B=-1), B.ATTN_ERR_INVALID_ARG),
    (dict(Lq=-5), B.ATTN_ERR_INVALID_ARG),
    (dict(D=96), B.ATTN_ERR_UNSUPPORTED),
    (dict(D=256), B.ATTN_ERR_UNSUPPORTED),
    (dict(causal=2), B.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), B.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), B.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("-inf")), B.ATTN_ERR_INVALID_ARG),
    (dict(q=FAKE + 8), B.ATTN_ERR_ALIGNMENT),
    (dict(out=FAKE + 2), B.ATTN_ERR_ALIGNMENT),
    (dict(lse=FAKE + 2), B.ATTN_ERR_ALIGNMENT),
])
def test_fwd_validation(lib, kw, code):
    assert fwd(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(kc=None), B.ATTN_ERR_INVALID_ARG),
    (dict(lens=None), B.ATTN_ERR_INVALID_ARG),
    (dict(Hq=6, Hkv=4), B.ATTN_ERR_INVALID_ARG),
    (dict(Lmax=-1), B.ATTN_ERR_INVALID_ARG),
    (dict(D=80), B.ATTN_ERR_UNSUPPORTED),
    (dict(vc=FAKE + 4), B.ATTN_ERR_ALIGNMENT),
    (dict(lens=FAKE + 2), B.ATTN_ERR_ALIGNMENT),
])
def test_decode_validation(lib, kw, code):
    assert dec(lib, **kw) == code


def test_varlen_validation(lib):
    p = B.attn_fwd_params()
    p.q = p.k = p.v = p.out = FAKE
    p.B, p.Hq, p.Hkv, p.Lq, p.Lkv, p.D = 2, 4, 4, 16, 16, 64
    p.scale, p.causal, p.total_q, p.total_k = 0.1, 1, 20, 20
    p.cu_seqlens_q = FAKE
    p.cu_seqlens_k = None  # one of the pair missing
    assert lib.attn_fwd_ex(ctypes.byref(p)) == B.ATTN_ERR_INVALID_ARG
    p.cu_seqlens_k = FAKE + 2
    assert lib.attn_fwd_ex(ctypes.byref(p)) == B.ATTN_ERR_ALIGNMENT
    p.cu_seqlens_k = FAKE
    p.out_dtype = 7
    assert lib.attn_fwd_ex(ctypes.byref(p)) == B.ATTN_ERR_INVALID_ARG


def test_decode_chunk_validation(lib):
    p = B.attn_decode_params()
    p.q = p.kcache = p.vcache = p.kv_lens = p.out = FAKE
    p.B, p.Hq, p.Hkv, p.Lmax, p.D, p.scale = 1, 4, 4, 128, 128, 0.1
    p.chunk = -64
    assert lib.attn_decode_ex(ctypes.byref(p)) == B.ATTN_ERR_INVALID_ARG


def multi(lib, **kw):
    p = B.attn_decode_multi_params()
    p.q = p.kcache = p.vcache = p.kv_lens = p.out = FAKE
    p.B, p.Hq, p.Hkv, p.Lq, p.Lmax, p.D, p.scale = 2, 8, 2, 4, 64, 128, 0.1
    for k, v in kw.items():
        setattr(p, k, v)
    return lib.attn_decode_multi(ctypes.byref(p))


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), B.ATTN_ERR_INVALID_ARG),
    (dict(kv_lens=None), B.ATTN_ERR_INVALID_ARG),
    (dict(Lq=0), B.ATTN_ERR_INVALID_ARG),
    (dict(Lq=-3), B.ATTN_ERR_INVALID_ARG),
    (dict(Hq=6, Hkv=4), B.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), B.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), B.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("-inf")), B.ATTN_ERR_INVALID_ARG),
    (dict(out_dtype=5), B.ATTN_ERR_INVALID_ARG),
    (dict(D=96), B.ATTN_ERR_UNSUPPORTED),
    (dict(Lq=33), B.ATTN_ERR_UNSUPPORTED),           # 4 heads x 33 tokens > one 128-row tile
    (dict(Hq=32, Hkv=2, Lq=9), B.ATTN_ERR_UNSUPPORTED),
    (dict(B=65535, Hkv=2, Hq=2, Lq=1), B.ATTN_ERR_UNSUPPORTED),  # more items than counter slots
    (dict(out=FAKE + 4), B.ATTN_ERR_ALIGNMENT),
    (dict(kv_lens=FAKE + 2), B.ATTN_ERR_ALIGNMENT),
])
def test_decode_multi_validation(lib, kw, code):
    assert multi(lib, **kw) == code


def test_selftest_limit_validation(lib):
    assert lib.attn_selftest_wait_timeout(0, None) == B.ATTN_ERR_INVALID_ARG
    assert lib.attn_selftest_wait_timeout(2000000, None) == B.ATTN_ERR_INVALID_ARG


def test_empty_inputs_are_noops(lib):
    assert fwd(lib, B=0) == B.ATTN_OK
    assert fwd(lib, Lq=0) == B.ATTN_OK
    assert dec(lib, B=0) == B.ATTN_OK
    assert multi(lib, B=0) == B.ATTN_OK


def test_no_cpu_fallback(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert fwd(lib) in (B.ATTN_ERR_UNSUPPORTED, B.ATTN_ERR_CUDA)
    assert dec(lib) in (B.ATTN_ERR_UNSUPPORTED, B.ATTN_ERR_CUDA)
    assert multi(lib) in (B.ATTN_ERR_UNSUPPORTED, B.ATTN_ERR_CUDA)


def test_workspace_bytes_formula(lib):
    import torch

    assert lib.attn_decode_workspace_bytes(0, 8, 2, 64, 128, 0) == 0
    assert lib.attn_decode_workspace_bytes(1, 8, 2, 64, 100, 0) == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 148
    grid = 3 * sms  # persistent decode: three CTAs per SM when a CTA serves 4 query heads
    # 256 KiB of counters + 2 partials per CTA x 4 heads per CTA x (D + 2) floats; independent of B, Lmax, chunk
    want = 65536 * 4 + 2 * grid * 4 * 130 * 4
    assert lib.attn_decode_workspace_bytes(2, 8, 2, 1000, 128, 256) == want
    assert lib.attn_decode_workspace_bytes(64, 8, 2, 99999, 128, 0) == want
    # too many rows for the counter area
    assert lib.attn_decode_workspace_bytes(65535, 64, 64, 16, 128, 0) == 0


def _fwd_params(**kw):
    p = B.attn_fwd_params()
    p.q = p.k = p.v = p.out = FAKE
    p.B, p.Hq, p.Hkv, p.Lq, p.Lkv, p.D = 1, 4, 2, 16, 16, 128
    p.scale, p.causal = 0.1, 1
    p.rope.cos, p.rope.sin, p.rope.max_pos, p.rope.style = FAKE, FAKE, 64, B.ATTN_ROPE_HALF
    for k, v in kw.items():
        if k.startswith("rope_"):
            setattr(p.rope, k[5:], v)
        else:
            setattr(p, k, v)
    return p


@pytest.mark.parametrize("kw,code", [
    (dict(rope_style=3), B.ATTN_ERR_INVALID_ARG),
    (dict(rope_sin=None), B.ATTN_ERR_INVALID_ARG),
    (dict(rope_max_pos=0), B.ATTN_ERR_INVALID_ARG),
    (dict(rope_max_pos=15), B.ATTN_ERR_INVALID_ARG),          # positions reach Lkv - 1 = 15
    (dict(rope_cos=FAKE + 4), B.ATTN_ERR_ALIGNMENT),
    (dict(Lq=32, Lkv=16), B.ATTN_ERR_INVALID_ARG),            # dense queries would sit before position 0
])
def test_fwd_rope_validation(lib, kw, code):
    assert lib.attn_fwd_ex(ctypes.byref(_fwd_params(**kw))) == code


def test_rope_off_when_style_none_or_no_table(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # no rotation requested: the bad table fields are not looked at (fails only for want of a device)
    for kw in (dict(rope_style=B.ATTN_ROPE_NONE, rope_max_pos=1), dict(rope_cos=None, rope_max_pos=1)):
        assert lib.attn_fwd_ex(ctypes.byref(_fwd_params(**kw))) in (B.ATTN_ERR_UNSUPPORTED, B.ATTN_ERR_CUDA)


def test_decode_rope_validation(lib):
    p = B.attn_decode_params()
    p.q = p.kcache = p.vcache = p.kv_lens = p.out = FAKE
    p.B, p.Hq, p.Hkv, p.Lmax, p.D, p.scale = 1, 4, 4, 128, 128, 0.1
    p.rope.cos, p.rope.sin, p.rope.max_pos, p.rope.style = FAKE, FAKE, 127, B.ATTN_ROPE_INTERLEAVED
    assert lib.attn_decode_ex(ctypes.byref(p)) == B.ATTN_ERR_INVALID_ARG  # kv_len may reach Lmax = 128
    assert lib.attn_decode_noalloc(ctypes.byref(p)) == B.ATTN_ERR_INVALID_ARG
    m = B.attn_decode_multi_params()
    m.q = m.kcache = m.vcache = m.kv_lens = m.out = FAKE
    m.B, m.Hq, m.Hkv, m.Lq, m.Lmax, m.D, m.scale = 1, 4, 4, 2, 128, 128, 0.1
    m.rope.cos, m.rope.sin, m.rope.max_pos, m.rope.style = FAKE, FAKE, 127, B.ATTN_ROPE_HALF
    assert lib.attn_decode_multi(ctypes.byref(m)) == B.ATTN_ERR_INVALID_ARG


def test_any_finite_scale_passes_validation(lib):
    # The scale multiplies the logits before the mask is added, and every finite value means something: 0 gives
    # uniform weights over the visible keys, a negative value reverses the order of the logits.  Validation lets
    # them through; here, with no sm_103 device, the calls then fail for want of one (never INVALID_ARG).
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present (the fake pointers must not reach a kernel)")
    for sc in (0.0, -0.0, -0.088, -3.5, 1e-30, -1e30):
        assert fwd(lib, scale=sc) in (B.ATTN_ERR_UNSUPPORTED, B.ATTN_ERR_CUDA), sc
        assert dec(lib, scale=sc) in (B.ATTN_ERR_UNSUPPORTED, B.ATTN_ERR_CUDA), sc
        assert multi(lib, scale=sc) in (B.ATTN_ERR_UNSUPPORTED, B.ATTN_ERR_CUDA), sc


def test_binding_refuses_wrong_output_shapes_and_devices():
    # Outputs are written over their full extent by the kernels: the binding compares every caller-supplied
    # buffer's shape and device with what the call will write, before any pointer reaches the library.
    import torch

    good = torch.empty(2, 3, 4)
    with pytest.raises(ValueError, match="shape"):
        B._need(torch.empty(2, 3, 5), "out", torch.float32, 3, (2, 3, 4))
    with pytest.raises(ValueError, match="dims"):
        B._need(torch.empty(2, 3), "out", torch.float32, 3, (2, 3, 4))
    with pytest.raises(TypeError):
        B._need(good, "out", torch.bfloat16, 3, (2, 3, 4))
    with pytest.raises(ValueError, match="CUDA"):  # right shape, but not on a GPU
        B._need(good, "out", torch.float32, 3, (2, 3, 4))
    p = B.attn_fwd_params()
    tab = torch.empty(8, 32)
    with pytest.raises(ValueError, match="shape"):  # rotated keys must be shaped like k
        B._set_rope(p, (tab, tab, "half", torch.empty(1, 2, 16, 64, dtype=torch.bfloat16)), 64,
                    torch.device("cpu"), (1, 2, 17, 64))
    with pytest.raises(ValueError, match="prefill"):  # decode calls take no k_out
        B._set_rope(p, (tab, tab, "half", torch.empty(1, 2, 16, 64, dtype=torch.bfloat16)), 64,
                    torch.device("cpu"))
