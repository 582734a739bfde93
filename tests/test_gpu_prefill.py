"""GPU parity of tensor-core prefill (attn_fwd / attn_fwd_ex) against the fp64 oracle.

Small shapes are compared element by element over every output; they cover
both head dims, causal and not, grouped heads, ragged last tiles, Lq != Lkv
in both directions (bottom-right causal alignment, rows that see no key), a
single query, a single key, no keys at all, fp32 output and logits large
enough to trigger the O rescale.  The prefill workloads run at full size in
the bench's launch configuration and are checked on sampled rows that the
oracle computes one by one, plus every row of one whole head (of the longest
sequence, for the packed workload); so are a shape with more work items than
SMs (every persistent CTA walks several jobs) and one 65,536-token sequence at
each head dim.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_attn_fwd_06_gb300 import binding as AB
from attention_attn_fwd_06_gb300.build import build
from attention_attn_fwd_06_gb300.inputs import WORKLOADS, make_prefill, make_varlen
from tests._parity import assert_attn_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    AB.load()
    AB.attn_get_device_status()
    yield
    assert AB.attn_get_device_status() == AB.ATTN_OK


def run(q, k, v, causal, scale=None, out_dtype=torch.bfloat16):
    out, lse = AB.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lkv,D,causal", [
    (1, 2, 2, 128, 128, 64, True),     # one full tile
    (1, 2, 2, 200, 200, 128, True),    # ragged last tile
    (2, 4, 2, 300, 300, 128, False),   # GQA, non-causal, three tiles
    (1, 4, 4, 100, 333, 128, True),    # Lq < Lkv: bottom-right causal offset
    (1, 2, 2, 333, 100, 64, True),     # Lq > Lkv: the first rows see no key
    (1, 8, 2, 513, 513, 64, True),     # GQA, D = 64, 5 tiles
    (1, 2, 1, 1, 77, 128, True),       # a single query row
    (1, 2, 2, 64, 1, 128, False),      # a single key
    (2, 2, 2, 256, 640, 128, False),   # several K tiles, exact multiples
    (1, 16, 1, 300, 300, 64, True),    # multi-query: 16 heads on one kv head
    (2, 16, 2, 200, 450, 128, False),  # 8 heads per kv head, Lq < Lkv, non-causal
])
def test_prefill_small(B, Hq, Hkv, Lq, Lkv, D, causal):
    q, k, v = make_prefill(B, Hq, Hkv, Lq, Lkv, D, seed=Lq * 7 + Lkv)
    scale = D ** -0.5
    O, lse = run(q, k, v, causal)
    O_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    assert_attn_close(O, lse, O_ref, lse_ref)


def test_prefill_tiny_workload_fp32():
    w = WORKLOADS["tiny_causal"]
    q, k, v = make_prefill(w.B, w.Hq, w.Hkv, w.L, w.L, w.D, w.seed)
    O, lse = run(q, k, v, True, out_dtype=torch.float32)
    assert O.dtype == torch.float32
    O_ref, lse_ref = oracle.attention(q, k, v, w.scale, True)
    assert_attn_close(O, lse, O_ref, lse_ref, "tiny_causal")


def test_prefill_no_keys():
    q, k, v = make_prefill(1, 2, 2, 50, 0, 128, seed=3)
    O, lse = run(q, k, v, False)
    assert torch.all(O == 0) and torch.all(torch.isneginf(lse))


def test_prefill_peaked_logits_rescale():
    q, k, v = make_prefill(1, 4, 4, 384, 384, 128, seed=9)
    q = (q.float() * 6).to(torch.bfloat16)
    k[:, :, 300:305] = (k[:, :, 300:305].float() * 3).to(torch.bfloat16)
    for causal in (False, True):
        O, lse = run(q, k, v, causal)
        O_ref, lse_ref = oracle.attention(q, k, v, 128 ** -0.5, causal)
        assert_attn_close(O, lse, O_ref, lse_ref, f"causal={causal}")


def test_prefill_custom_scale():
    q, k, v = make_prefill(1, 2, 2, 130, 130, 64, seed=21)
    O, lse = run(q, k, v, True, scale=0.37)
    O_ref, lse_ref = oracle.attention(q, k, v, 0.37, True)
    assert_attn_close(O, lse, O_ref, lse_ref)


def test_prefill_deterministic():
    q, k, v = make_prefill(1, 4, 2, 700, 700, 128, seed=31)
    a = run(q, k, v, True)
    b = run(q, k, v, True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D", [64, 128])
def test_prefill_varlen_small(causal, D):
    q, k, v, cu = make_varlen(4, 8, 2, D, seed=41 + D, seqlens=[5, 130, 1, 260])
    out, lse = AB.attn_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cu.to(DEV), cu.to(DEV), 260, 260, causal=causal)
    torch.cuda.synchronize()
    O_ref, lse_ref = oracle.attention_varlen(q, k, v, cu.tolist(), cu.tolist(), D ** -0.5, causal)
    assert_attn_close(out.cpu(), lse.cpu(), O_ref, lse_ref)


def test_prefill_varlen_empty_sequence_and_fp32():
    q, k, v, cu = make_varlen(3, 4, 4, 128, seed=43, seqlens=[70, 0, 129])
    out, lse = AB.attn_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cu.to(DEV), cu.to(DEV), 129, 129, causal=True,
                                  out_dtype=torch.float32)
    torch.cuda.synchronize()
    O_ref, lse_ref = oracle.attention_varlen(q, k, v, cu.tolist(), cu.tolist(), 128 ** -0.5, True)
    assert_attn_close(out.cpu(), lse.cpu(), O_ref, lse_ref)


def test_decode_equals_last_row_of_prefill_on_gpu():
    # The same data through both entry points: decode over L keys == row L-1 of causal prefill.
    q, k, v = make_prefill(1, 8, 2, 300, 300, 128, seed=51)
    Op, lsep = run(q, k, v, True)
    qd = q[:, :, -1].contiguous()
    lens = torch.tensor([300], dtype=torch.int32, device=DEV)
    Od, lsed = AB.attn_decode(qd.to(DEV), k.to(DEV), v.to(DEV), lens)
    torch.cuda.synchronize()
    assert_attn_close(Od.cpu(), lsed.cpu(), Op[:, :, -1].double().numpy(), lsep[:, :, -1].double().numpy())


def _sample_rows(rng, L, n):
    rows = set(rng.choice(L, size=min(n, L), replace=False).tolist())
    rows |= {0, L - 1, min(127, L - 1), min(128, L - 1)}
    return np.array(sorted(rows))


def _every_row(L, step=1024):
    return [np.arange(r0, min(L, r0 + step)) for r0 in range(0, L, step)]


@pytest.mark.parametrize("name", ["prefill_causal", "prefill_noncausal_d64"])
def test_prefill_workload_sampled(name):
    # Sampled rows of three heads per batch entry, and then EVERY row of one whole head (the last batch entry's
    # last head: every (query tile, key tile) pair of that head, the diagonal and the last tiles included),
    # element by element against the oracle in blocks of rows.
    w = WORKLOADS[name]
    q, k, v = make_prefill(w.B, w.Hq, w.Hkv, w.L, w.L, w.D, w.seed)
    O, lse = run(q, k, v, w.causal)
    assert torch.isfinite(O.float()).all() and torch.isfinite(lse).all()
    rng = np.random.default_rng(7)
    for b in range(w.B):
        for h in rng.choice(w.Hq, 3, replace=False):
            rows = _sample_rows(rng, w.L, 48)
            O_ref, lse_ref = oracle.attention_rows(q, k, v, w.scale, w.causal, b, int(h), rows)
            assert_attn_close(O[b, h, rows], lse[b, h, rows], O_ref, lse_ref, f"{name} b={b} h={h}")
    b, h = w.B - 1, w.Hq - 1
    for rows in _every_row(w.L):
        O_ref, lse_ref = oracle.attention_rows(q, k, v, w.scale, w.causal, b, h, rows)
        assert_attn_close(O[b, h, rows], lse[b, h, rows], O_ref, lse_ref, f"{name} full head b={b} h={h}")


@pytest.mark.parametrize("D,causal", [(128, True), (64, False)])
def test_prefill_64k_sequence_sampled(D, causal):
    """One 65,536-token sequence (8x the longest workload), grouped heads: sampled rows across the whole range,
    the last rows included, against the oracle row by row."""
    B, Hq, Hkv, L = 1, 2, 1, 65536
    q, k, v = make_prefill(B, Hq, Hkv, L, L, D, seed=65536 + D)
    O, lse = run(q, k, v, causal)
    assert torch.isfinite(O.float()).all() and torch.isfinite(lse).all()
    rng = np.random.default_rng(13)
    for h in range(Hq):
        rows = _sample_rows(rng, L, 24)
        rows = np.union1d(rows, [L - 129, L - 128, L - 2])
        O_ref, lse_ref = oracle.attention_rows(q, k, v, D ** -0.5, causal, 0, h, rows)
        assert_attn_close(O[0, h, rows], lse[0, h, rows], O_ref, lse_ref, f"L={L} D={D} h={h}")


def test_prefill_ragged_workload_sampled():
    w = WORKLOADS["prefill_ragged_gqa"]
    q, k, v, cu = make_varlen(w.B, w.Hq, w.Hkv, w.D, w.seed, seq_range=w.seq_range)
    lens = (cu[1:] - cu[:-1]).tolist()
    mx = max(lens)
    out, lse = AB.attn_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cu.to(DEV), cu.to(DEV), mx, mx, causal=True)
    torch.cuda.synchronize()
    out, lse = out.cpu(), lse.cpu()
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    rng = np.random.default_rng(11)
    cul = cu.tolist()
    for s in range(w.B):
        h = int(rng.integers(w.Hq))
        rows = _sample_rows(rng, lens[s], 24)
        O_ref, lse_ref = oracle.attention_varlen_rows(q, k, v, cul, cul, w.scale, True, s, h, rows)
        idx = torch.as_tensor(cul[s] + rows)
        assert_attn_close(out[idx, h], lse[idx, h], O_ref, lse_ref, f"seq {s} (len {lens[s]}) h={h}")
    # every row of one head of the longest sequence (the last query head: the last kv head's group)
    s = int(np.argmax(lens))
    h = w.Hq - 1
    for rows in _every_row(lens[s]):
        O_ref, lse_ref = oracle.attention_varlen_rows(q, k, v, cul, cul, w.scale, True, s, h, rows)
        idx = torch.as_tensor(cul[s] + rows)
        assert_attn_close(out[idx, h], lse[idx, h], O_ref, lse_ref, f"longest seq {s} (len {lens[s]}) full head")


@pytest.mark.parametrize("D,causal", [(128, False), (128, True), (64, False)])
def test_prefill_persistent_many_items(D, causal):
    # More work items than SMs (B * Hq * tile pairs = 2 * 32 * 5 = 320 non-causal), so every persistent CTA walks
    # several jobs; GQA 4:1 and a ragged last tile (1200 = 9 * 128 + 48); sampled rows of every head checked
    B, Hq, Hkv, L = 2, 32, 8, 1200
    q, k, v = make_prefill(B, Hq, Hkv, L, L, D, seed=90 + D + causal)
    O, lse = run(q, k, v, causal)
    assert torch.isfinite(O.float()).all() and torch.isfinite(lse).all()
    rng = np.random.default_rng(D + causal)
    for b in range(B):
        for h in range(0, Hq, 5):
            rows = np.array(sorted(set(rng.choice(L, 6, replace=False).tolist()) | {0, L - 1}))
            O_ref, lse_ref = oracle.attention_rows(q, k, v, D ** -0.5, causal, b, h, rows)
            assert_attn_close(O[b, h, rows], lse[b, h, rows], O_ref, lse_ref, f"b={b} h={h}")


@pytest.mark.parametrize("D", [64, 128])
def test_prefill_fault_injection_times_out_and_recovers(monkeypatch, D):
    # ATTN_FAULT_INJECT=skip_arrive: one softmax thread of CTA 0 withholds its P-ready arrival for the second K
    # step of its first tile; the MMA warp's bounded wait runs out (about a second), every role of that CTA winds
    # down (in-flight copies and MMAs drained, TMEM freed), the status word reports the timeout, and the next
    # clean call is correct.  Both warp layouts: D = 64 (10 warps) and D = 128 (12 warps, register split).
    q, k, v = make_prefill(1, 2, 2, 512, 512, D, seed=77 + D)  # CTA 0's first tile pair has 4 K steps
    AB.attn_get_device_status()
    monkeypatch.setenv("ATTN_FAULT_INJECT", "skip_arrive")
    run(q, k, v, False)
    assert AB.attn_get_device_status() == AB.ATTN_ERR_DEVICE_TIMEOUT
    monkeypatch.delenv("ATTN_FAULT_INJECT")
    O, lse = run(q, k, v, False)
    assert AB.attn_get_device_status() == AB.ATTN_OK
    O_ref, lse_ref = oracle.attention(q, k, v, D ** -0.5, False)
    assert_attn_close(O, lse, O_ref, lse_ref)
