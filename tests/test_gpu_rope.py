"""GPU parity of the fused rotary position embedding against the fp64 oracle.

Prefill rotates the keys (optionally into a caller buffer, which is checked
too) and the queries once per call, in a pass each, before the attention
kernel; the decode kernels rotate only the query (the cache holds
keys already rotated, so any cache contents serve).  Both pair layouts, both
head dims, Lq < Lkv (queries placed at Lkv - Lq + i), packed sequences, paged
caches, multi-token decode and the causal prefill workload at full size
(sampled rows) are covered.  Tables come from the standard frequency ladder.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_attn_fwd_06_gb300 import binding as AB
from attention_attn_fwd_06_gb300.build import build
from attention_attn_fwd_06_gb300.inputs import (WORKLOADS, make_decode, make_decode_multi, make_pages, make_prefill,
                                                make_varlen, rope_tables)
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


def tables(max_pos, D):
    cos, sin = rope_tables(max_pos, D)
    return cos, sin, cos.to(DEV), sin.to(DEV)


@pytest.mark.parametrize("style", ["half", "interleaved"])
@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lkv,D,causal", [
    (1, 2, 2, 200, 200, 128, True),    # ragged last tile
    (2, 4, 2, 300, 300, 128, False),   # GQA, non-causal
    (1, 4, 4, 100, 333, 128, True),    # Lq < Lkv: queries sit at 233 ..
    (1, 8, 2, 513, 513, 64, True),     # D = 64
])
def test_prefill_rope_small(style, B, Hq, Hkv, Lq, Lkv, D, causal):
    q, k, v = make_prefill(B, Hq, Hkv, Lq, Lkv, D, seed=Lq + 3 * Lkv)
    cos, sin, cos_d, sin_d = tables(Lkv + 50, D)
    O, lse = AB.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, rope=(cos_d, sin_d, style))
    torch.cuda.synchronize()
    O_ref, lse_ref = oracle.attention(q, k, v, D ** -0.5, causal, rope=(cos, sin, style))
    assert_attn_close(O.cpu(), lse.cpu(), O_ref, lse_ref)


@pytest.mark.parametrize("style", ["half", "interleaved"])
def test_prefill_rope_varlen(style):
    q, k, v, cu = make_varlen(4, 8, 2, 128, seed=61, seqlens=[5, 130, 1, 260])
    cos, sin, cos_d, sin_d = tables(300, 128)
    out, lse = AB.attn_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cu.to(DEV), cu.to(DEV), 260, 260, causal=True,
                                  rope=(cos_d, sin_d, style))
    torch.cuda.synchronize()
    O_ref, lse_ref = oracle.attention_varlen(q, k, v, cu.tolist(), cu.tolist(), 128 ** -0.5, True,
                                             rope=(cos, sin, style))
    assert_attn_close(out.cpu(), lse.cpu(), O_ref, lse_ref)


@pytest.mark.parametrize("style", ["half", "interleaved"])
def test_prefill_rope_varlen_fewer_queries_than_keys(style):
    # each packed sequence places its queries at Lkv_s - Lq_s + i: the query pass shifts every sequence by its own
    # offset (0, 66, 6 and 160 here)
    q_lens, k_lens = [5, 64, 1, 100], [5, 130, 7, 260]
    q, _, _, cu_q = make_varlen(4, 8, 2, 128, seed=71, seqlens=q_lens)
    _, k, v, cu_k = make_varlen(4, 8, 2, 128, seed=72, seqlens=k_lens)
    cos, sin, cos_d, sin_d = tables(300, 128)
    AB.attn_get_device_status()
    out, lse = AB.attn_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cu_q.to(DEV), cu_k.to(DEV), max(q_lens),
                                  max(k_lens), causal=True, rope=(cos_d, sin_d, style))
    torch.cuda.synchronize()
    assert AB.attn_get_device_status() == AB.ATTN_OK
    O_ref, lse_ref = oracle.attention_varlen(q, k, v, cu_q.tolist(), cu_k.tolist(), 128 ** -0.5, True,
                                             rope=(cos, sin, style))
    assert_attn_close(out.cpu(), lse.cpu(), O_ref, lse_ref)


def test_prefill_rope_varlen_more_queries_than_keys_is_flagged():
    # a packed sequence with more queries than keys would place its first queries before position 0: the call
    # reports ATTN_ERR_DEVICE_BOUNDS (its rows are then not meaningful) and the other sequences are unaffected
    q_lens, k_lens = [40, 64], [64, 20]
    q, _, _, cu_q = make_varlen(2, 4, 2, 128, seed=73, seqlens=q_lens)
    _, k, v, cu_k = make_varlen(2, 4, 2, 128, seed=74, seqlens=k_lens)
    cos, sin, cos_d, sin_d = tables(100, 128)
    AB.attn_get_device_status()
    out, lse = AB.attn_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cu_q.to(DEV), cu_k.to(DEV), 64, 64,
                                  causal=True, rope=(cos_d, sin_d, "half"))
    torch.cuda.synchronize()
    assert AB.attn_get_device_status() == AB.ATTN_ERR_DEVICE_BOUNDS
    O_ref, lse_ref = oracle.attention_varlen(q[:40], k[:64], v[:64], [0, 40], [0, 64], 128 ** -0.5, True,
                                             rope=(cos, sin, "half"))
    assert_attn_close(out[:40].cpu(), lse[:40].cpu(), O_ref, lse_ref)
    assert AB.attn_get_device_status() == AB.ATTN_OK


def test_prefill_rope_writes_rotated_keys():
    # k_out receives the rotated keys (what a serving engine appends to its cache): the oracle's rotation held in
    # bf16, up to a last-bit difference where fp32 and fp64 arithmetic round to different neighbours
    q, k, v = make_prefill(2, 4, 2, 300, 300, 128, seed=5)
    cos, sin, cos_d, sin_d = tables(300, 128)
    k_out = torch.empty_like(k, device=DEV)
    O, lse = AB.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, rope=(cos_d, sin_d, "half", k_out))
    torch.cuda.synchronize()
    want = oracle.round_bf16(oracle.rope_rotate(k, np.arange(300), cos, sin, "half"))
    got = k_out.cpu().double().numpy()
    ulp = np.abs(want) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(got - want) <= ulp), "rotated keys off by more than one bf16 step"
    assert np.mean(got != want) < 1e-3
    O_ref, lse_ref = oracle.attention(q, k, v, 128 ** -0.5, True, rope=(cos, sin, "half"))
    assert_attn_close(O.cpu(), lse.cpu(), O_ref, lse_ref)


def test_prefill_rope_rejects_short_tables():
    q, k, v = make_prefill(1, 2, 2, 64, 64, 128, seed=1)
    _, _, cos_d, sin_d = tables(63, 128)
    with pytest.raises(AB.AttnError) as e:
        AB.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, rope=(cos_d, sin_d, "half"))
    assert e.value.status == AB.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("style", ["half", "interleaved"])
@pytest.mark.parametrize("D", [64, 128])
def test_decode_rope(style, D):
    q, kc, vc, _ = make_decode(3, 16, 4, 513, D, seed=71 + D)
    lens = [513, 64, 1]
    cos, sin, cos_d, sin_d = tables(600, D)
    out, lse = AB.attn_decode(q.to(DEV), kc.to(DEV), vc.to(DEV), torch.tensor(lens, dtype=torch.int32, device=DEV),
                              rope=(cos_d, sin_d, style))
    torch.cuda.synchronize()
    O_ref, lse_ref = oracle.decode(q, kc, vc, lens, D ** -0.5, rope=(cos, sin, style))
    assert_attn_close(out.cpu(), lse.cpu(), O_ref, lse_ref)


def test_decode_paged_rope():
    q, kc, vc, _ = make_decode(2, 32, 8, 700, 128, seed=73)
    lens = [700, 333]
    kp, vp, table = make_pages(kc, vc, 16, seed=74)
    cos, sin, cos_d, sin_d = tables(704, 128)
    out, lse = AB.attn_decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV),
                                    torch.tensor(lens, dtype=torch.int32, device=DEV), rope=(cos_d, sin_d, "half"))
    torch.cuda.synchronize()
    O_ref, lse_ref = oracle.decode(q, kc, vc, lens, 128 ** -0.5, rope=(cos, sin, "half"))
    assert_attn_close(out.cpu(), lse.cpu(), O_ref, lse_ref)


@pytest.mark.parametrize("style", ["half", "interleaved"])
def test_decode_multi_rope(style):
    q, kc, vc, _ = make_decode_multi(3, 16, 4, 4, 600, 128, seed=79)
    lens = [600, 130, 3]  # the last: kv_len < Lq, its first token sees no key and is not rotated
    cos, sin, cos_d, sin_d = tables(600, 128)
    out, lse = AB.attn_decode_multi(q.to(DEV), kc.to(DEV), vc.to(DEV),
                                    torch.tensor(lens, dtype=torch.int32, device=DEV), rope=(cos_d, sin_d, style))
    torch.cuda.synchronize()
    O_ref, lse_ref = oracle.decode_multi(q, kc, vc, lens, 128 ** -0.5, rope=(cos, sin, style))
    assert_attn_close(out.cpu(), lse.cpu(), O_ref, lse_ref)


def test_prefill_rope_workload_sampled():
    w = WORKLOADS["prefill_causal"]
    q, k, v = make_prefill(w.B, w.Hq, w.Hkv, w.L, w.L, w.D, w.seed)
    cos, sin, cos_d, sin_d = tables(w.L, w.D)
    O, lse = AB.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, rope=(cos_d, sin_d, "half"))
    torch.cuda.synchronize()
    O, lse = O.cpu(), lse.cpu()
    rng = np.random.default_rng(17)
    for b in range(w.B):
        h = int(rng.integers(w.Hq))
        rows = np.array(sorted(set(rng.choice(w.L, 24, replace=False).tolist()) | {0, w.L - 1}))
        O_ref, lse_ref = oracle.attention_rows(q, k, v, w.scale, True, b, h, rows, rope=(cos, sin, "half"))
        assert_attn_close(O[b, h, rows], lse[b, h, rows], O_ref, lse_ref, f"b={b} h={h}")
