"""The decode entry point that allocates no device memory (attn_decode_noalloc).

Some callers cannot let a library call cudaMalloc: code running under CUDA
graph capture, serving engines that hand all of HBM to their own pool, and
latency paths that cannot absorb cudaMalloc's synchronisation.  For them the
library offers attn_decode_noalloc, which keeps its split-KV partials in a
fixed buffer compiled into the library instead of a workspace it allocates.

These tests call it through the C ABI and check its output against the
regular attn_decode_ex entry point on the same inputs, for two calls in a row
(the second call finds the buffer holding the first call's contents), a
call captured into a CUDA graph and replayed on new data, and (in a fresh
process) that a first call made inside a stream capture is refused without
spoiling the capture.  The
file sorts last so a run that stops at the first failure has already run
every other test.
"""
import ctypes
import os
import subprocess
import sys
import textwrap

import pytest
import torch

from attention_attn_fwd_06_gb300 import binding as AB
from attention_attn_fwd_06_gb300.build import build
from attention_attn_fwd_06_gb300.inputs import make_decode
from tests._parity import assert_attn_close


@pytest.fixture(scope="module")
def lib():
    build()
    return AB.load()


def test_noalloc_symbol_exported(lib):
    assert hasattr(lib, "attn_decode_noalloc")
    assert AB.status_string(AB.ATTN_ERR_SCRATCH_TOO_SMALL) == "ATTN_ERR_SCRATCH_TOO_SMALL"


def test_noalloc_rejects_problem_beyond_scratch(lib):
    # The fixed buffer's counter area holds 65534 (b, kv head, head group) rows:
    # 16384 sequences x 8 kv heads x 1 group (4 heads per CTA) is too many.
    # Nothing is enqueued (the pointers are never dereferenced).
    p = AB.attn_decode_params()
    fake = 1 << 20
    p.q = p.kcache = p.vcache = p.kv_lens = p.out = fake
    p.B, p.Hq, p.Hkv, p.Lmax, p.D, p.scale = 16384, 32, 8, 64, 128, 0.088
    rc = lib.attn_decode_noalloc(ctypes.byref(p))
    if torch.cuda.is_available() and torch.cuda.get_device_capability() == (10, 3):
        assert rc == AB.ATTN_ERR_SCRATCH_TOO_SMALL
    else:  # no GPU, or a GPU the library does not support: refused before the size check
        assert rc in (AB.ATTN_ERR_UNSUPPORTED, AB.ATTN_ERR_CUDA)


@pytest.mark.gpu
@pytest.mark.parametrize("B,Hq,Hkv,Lmax,D,kv_range", [
    (8, 32, 8, 4096, 128, (512, 4096)),   # the GQA decode workload's shape
    (3, 16, 16, 777, 64, (1, 777)),       # D = 64, MHA, ragged lengths
])
def test_noalloc_matches_decode_ex_twice(lib, B, Hq, Hkv, Lmax, D, kv_range):
    dev = torch.device("cuda:0")
    results = []
    for call, seed in enumerate((71, 72)):  # two calls in a row with different data
        q, kc, vc, lens = make_decode(B, Hq, Hkv, Lmax, D, seed=seed + Lmax, kv_range=kv_range)
        q, kc, vc, lens = (t.to(dev) for t in (q, kc, vc, lens))
        ref_o, ref_lse = AB.attn_decode(q, kc, vc, lens)
        out = torch.empty_like(ref_o)
        lse = torch.empty_like(ref_lse)
        AB.attn_decode_noalloc(q, kc, vc, lens, out, lse)
        torch.cuda.synchronize()
        assert AB.attn_get_device_status() == AB.ATTN_OK
        assert_attn_close(out.cpu(), lse.cpu(), ref_o.double().cpu().numpy(), ref_lse.double().cpu().numpy(),
                          f"call {call}")
        results.append(out.cpu())
    assert not torch.equal(results[0], results[1])  # the second call really recomputed


@pytest.mark.gpu
def test_noalloc_replays_from_cuda_graph(lib):
    # The call a graph-captured decode step makes: capture once, then replay with new queries, cache contents and
    # lengths written in place -- each replay must match attn_decode_ex on that replay's data.
    dev = torch.device("cuda:0")
    B, Hq, Hkv, Lmax, D = 4, 32, 8, 2048, 128
    q, kc, vc, lens = (t.to(dev) for t in make_decode(B, Hq, Hkv, Lmax, D, seed=81, kv_range=(1, Lmax)))
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    AB.attn_decode_noalloc(q, kc, vc, lens, out, lse)  # first call on the device: outside any capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        AB.attn_decode_noalloc(q, kc, vc, lens, out, lse)
    for seed in (82, 83):
        q2, kc2, vc2, lens2 = make_decode(B, Hq, Hkv, Lmax, D, seed=seed, kv_range=(1, Lmax))
        q.copy_(q2)
        kc.copy_(kc2)
        vc.copy_(vc2)
        lens.copy_(lens2)
        g.replay()
        ref_o, ref_lse = AB.attn_decode(q, kc, vc, lens)
        torch.cuda.synchronize()
        assert AB.attn_get_device_status() == AB.ATTN_OK
        assert_attn_close(out.cpu(), lse.cpu(), ref_o.double().cpu().numpy(), ref_lse.double().cpu().numpy(),
                          f"replay seed {seed}")


_FIRST_CALL_IN_CAPTURE = textwrap.dedent("""
    import torch
    from attention_attn_fwd_06_gb300 import binding as AB
    from attention_attn_fwd_06_gb300.inputs import make_decode
    dev = torch.device("cuda:0")
    q, kc, vc, lens = (t.to(dev) for t in make_decode(2, 8, 2, 256, 128, seed=91, kv_range=(1, 256)))
    out = torch.zeros(2, 8, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(2, 8, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    refused = None
    with torch.cuda.graph(g):
        out.add_(1.0)
        try:
            AB.attn_decode_noalloc(q, kc, vc, lens, out, lse)
        except AB.AttnError as e:
            refused = e.status
    assert refused == AB.ATTN_ERR_INVALID_ARG, refused
    g.replay()  # the capture survived: its one op runs
    torch.cuda.synchronize()
    assert bool((out == 1.0).all())
    AB.attn_decode_noalloc(q, kc, vc, lens, out, lse)  # outside the capture the first call succeeds
    ref_o, ref_lse = AB.attn_decode(q, kc, vc, lens)
    torch.cuda.synchronize()
    assert AB.attn_get_device_status() == AB.ATTN_OK
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_lse)
    print("ok")
""")


@pytest.mark.gpu
def test_noalloc_first_call_inside_capture_is_refused(lib):
    # Needs a process where the entry point has not run yet on the device: a child interpreter.
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL_IN_CAPTURE], cwd=root, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]
