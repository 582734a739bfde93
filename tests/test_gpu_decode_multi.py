"""GPU parity of multi-token decode (attn_decode_multi) against the fp64 oracle.

Every small case fills the cache rows at or past kv_len with NaN, so a read of
them would poison O.  The cases cover both head dims, every query-row count
from 1 to a full 128-row tile (heads per kv head x tokens), lengths that are
exact tile multiples, one past them, shorter than a tile, shorter than Lq
(tokens that see no key) and zero, one long sequence split over every CTA
(many partials per item, merged in the kernel), fp32 output, logits peaked
enough to force the O rescale, determinism, Lq = 1 against the single-token
decode; the 8 x 4096 multi-token workload runs at full size with every row
checked, the 131k-key one and a 2^20-key cache on sampled heads (both ends of
several kv-head groups).
"""
import numpy as np
import pytest
import torch

import oracle
from attention_attn_fwd_06_gb300 import binding as AB
from attention_attn_fwd_06_gb300.build import build
from attention_attn_fwd_06_gb300.inputs import WORKLOADS, make_decode_multi
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


def poison_past_lens(kc, vc, lens):
    kc, vc = kc.clone(), vc.clone()
    for b, n in enumerate(lens):
        kc[b, :, n:] = float("nan")
        vc[b, :, n:] = float("nan")
    return kc, vc


def run(q, kc, vc, lens, scale=None, out_dtype=torch.bfloat16):
    out, lse = AB.attn_decode_multi(q.to(DEV), kc.to(DEV), vc.to(DEV), torch.as_tensor(lens, dtype=torch.int32).to(DEV),
                                    scale=scale, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lmax,D,lens", [
    (3, 16, 4, 4, 300, 128, [300, 129, 5]),     # 4 heads x 4 tokens; ragged tail, one short sequence
    (2, 32, 8, 8, 512, 128, [256, 257]),        # the workload's grouping; exact tile multiple and one past
    (2, 8, 8, 16, 200, 128, [200, 16]),         # MHA, 16 tokens; a sequence of exactly Lq keys
    (1, 16, 2, 16, 384, 128, [384]),            # 8 heads x 16 tokens = a full 128-row tile
    (2, 8, 2, 3, 140, 64, [140, 77]),           # D = 64, 12 rows
    (2, 16, 4, 2, 1000, 64, [1000, 640]),       # D = 64, several tiles
    (3, 8, 4, 8, 64, 128, [5, 0, 64]),          # kv_len < Lq (early tokens see nothing) and kv_len = 0
    (2, 4, 2, 1, 333, 128, [333, 1]),           # Lq = 1
])
def test_decode_multi_small(B, Hq, Hkv, Lq, Lmax, D, lens):
    q, kc, vc, _ = make_decode_multi(B, Hq, Hkv, Lq, Lmax, D, seed=17 + Lmax + Lq)
    kc, vc = poison_past_lens(kc, vc, lens)
    scale = D ** -0.5
    O, lse = run(q, kc, vc, lens)
    O_ref, lse_ref = oracle.decode_multi(q, kc, vc, lens, scale)
    assert_attn_close(O, lse, O_ref, lse_ref)


def test_decode_multi_many_sequences():
    # More sequences than a warp has lanes: the work walk's prefix sums take two passes of 32.
    B = 45
    g = torch.Generator().manual_seed(45)
    lens = torch.randint(0, 400, (B,), generator=g, dtype=torch.int32).tolist()
    lens[7] = 0
    lens[30] = 2  # fewer keys than new tokens
    q, kc, vc, _ = make_decode_multi(B, 16, 4, 4, 400, 128, seed=61)
    kc, vc = poison_past_lens(kc, vc, lens)
    O, lse = run(q, kc, vc, lens)
    O_ref, lse_ref = oracle.decode_multi(q, kc, vc, lens, 128 ** -0.5)
    assert_attn_close(O, lse, O_ref, lse_ref)


def test_decode_multi_long_sequence_split_over_all_ctas():
    # One item of 64 tiles on a grid of one CTA per SM: every CTA holds a piece, the last one merges them all.
    q, kc, vc, _ = make_decode_multi(1, 4, 1, 8, 8192, 128, seed=23)
    lens = [8192 - 37]
    kc, vc = poison_past_lens(kc, vc, lens)
    O, lse = run(q, kc, vc, lens)
    O_ref, lse_ref = oracle.decode_multi(q, kc, vc, lens, 128 ** -0.5)
    assert_attn_close(O, lse, O_ref, lse_ref)


def test_decode_multi_mixed_lengths_many_items():
    # Items of very different lengths: shares start and end inside items and span several whole items.
    lens = [4000, 1, 130, 0, 2048, 700, 3, 4096, 128, 2500]
    q, kc, vc, _ = make_decode_multi(len(lens), 16, 4, 4, 4096, 128, seed=29)
    kc, vc = poison_past_lens(kc, vc, lens)
    O, lse = run(q, kc, vc, lens, out_dtype=torch.float32)
    assert O.dtype == torch.float32
    O_ref, lse_ref = oracle.decode_multi(q, kc, vc, lens, 128 ** -0.5)
    assert_attn_close(O, lse, O_ref, lse_ref)


def test_decode_multi_peaked_logits_rescale():
    q, kc, vc, _ = make_decode_multi(2, 8, 2, 4, 1024, 128, seed=31)
    q = (q.float() * 5).to(torch.bfloat16)
    kc[:, :, 700:705] = (kc[:, :, 700:705].float() * 3).to(torch.bfloat16)  # late keys dominate
    lens = [1024, 900]
    O, lse = run(q, kc, vc, lens)
    O_ref, lse_ref = oracle.decode_multi(q, kc, vc, lens, 128 ** -0.5)
    assert_attn_close(O, lse, O_ref, lse_ref)


def test_decode_multi_deterministic():
    lens = [3000, 1500, 2222]
    q, kc, vc, _ = make_decode_multi(3, 32, 8, 8, 3072, 128, seed=37)
    a = run(q, kc, vc, lens)
    b = run(q, kc, vc, lens)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_decode_multi_one_token_matches_single_decode():
    q, kc, vc, _ = make_decode_multi(2, 16, 4, 1, 700, 128, seed=41)
    lens = torch.tensor([700, 301], dtype=torch.int32)
    Om, lsem = run(q, kc, vc, lens.tolist())
    Od, lsed = AB.attn_decode(q[:, :, 0].contiguous().to(DEV), kc.to(DEV), vc.to(DEV), lens.to(DEV))
    torch.cuda.synchronize()
    O_ref, lse_ref = oracle.decode(q[:, :, 0], kc, vc, lens.tolist(), 128 ** -0.5)
    assert_attn_close(Om[:, :, 0], lsem[:, :, 0], O_ref, lse_ref, "multi")
    assert_attn_close(Od.cpu(), lsed.cpu(), O_ref, lse_ref, "single")


def test_decode_multi_kv_len_out_of_range_is_flagged():
    q, kc, vc, _ = make_decode_multi(2, 4, 2, 2, 96, 128, seed=43)
    O, lse = run(q, kc, vc, [96, 500])  # 500 > Lmax: clamped to 96 and flagged
    assert AB.attn_get_device_status() == AB.ATTN_ERR_DEVICE_BOUNDS
    O_ref, lse_ref = oracle.decode_multi(q, kc, vc, [96, 96], 128 ** -0.5)
    assert_attn_close(O, lse, O_ref, lse_ref)


def test_decode_multi_rejects_too_many_rows():
    q = torch.zeros((1, 32, 9, 128), dtype=torch.bfloat16, device=DEV)  # 16 heads x 9 tokens = 144 rows
    kc = torch.zeros((1, 2, 64, 128), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(AB.AttnError) as e:
        AB.attn_decode_multi(q, kc, kc, torch.tensor([64], dtype=torch.int32, device=DEV))
    assert e.value.status == AB.ATTN_ERR_UNSUPPORTED


def test_decode_multi_workload_full():
    # Every (sequence, query head, token) row of the 8-token GQA workload against the oracle.
    w = WORKLOADS["decode_multi_gqa"]
    q, kc, vc, lens = make_decode_multi(w.B, w.Hq, w.Hkv, w.Lq, w.L, w.D, w.seed, kv_range=w.kv_range)
    O, lse = run(q, kc, vc, lens.tolist())
    assert torch.isfinite(O.float()).all() and torch.isfinite(lse).all()
    O_ref, lse_ref = oracle.decode_multi(q, kc, vc, lens.tolist(), w.scale)
    assert_attn_close(O, lse, O_ref, lse_ref, "decode_multi_gqa")


def test_decode_multi_long_workload_sampled():
    w = WORKLOADS["decode_multi_long"]
    q, kc, vc, lens = make_decode_multi(w.B, w.Hq, w.Hkv, w.Lq, w.L, w.D, w.seed, kv_lens=w.kv_lens)
    O, lse = run(q, kc, vc, lens.tolist())
    assert torch.isfinite(O.float()).all() and torch.isfinite(lse).all()
    heads = [(b, h) for b in range(w.B) for h in (0, 3, 4, 13, 18, 27, 28, 31)]  # both ends of several kv groups
    O_ref, lse_ref = oracle.decode_multi(q, kc, vc, lens.tolist(), w.scale, heads=heads)
    idx_b = [b for b, _ in heads]
    idx_h = [h for _, h in heads]
    assert_attn_close(O[idx_b, idx_h], lse[idx_b, idx_h], O_ref[idx_b, idx_h], lse_ref[idx_b, idx_h])


def test_decode_multi_million_key_cache_sampled():
    """4 new tokens over a 2^20-key cache (8x the longest workload) and one of 777,777 keys, sampled heads."""
    B, Hq, Hkv, Lq, Lmax, D = 2, 8, 2, 4, 1 << 20, 128
    q, kc, vc, lens = make_decode_multi(B, Hq, Hkv, Lq, Lmax, D, seed=(1 << 20) + 1, kv_lens=[Lmax, 777_777])
    O, lse = run(q, kc, vc, lens.tolist())
    assert torch.isfinite(O.float()).all() and torch.isfinite(lse).all()
    heads = [(0, 1), (0, 6), (1, 0), (1, 7)]
    O_ref, lse_ref = oracle.decode_multi(q, kc, vc, lens.tolist(), D ** -0.5, heads=heads)
    idx_b = [b for b, _ in heads]
    idx_h = [h for _, h in heads]
    assert_attn_close(O[idx_b, idx_h], lse[idx_b, idx_h], O_ref[idx_b, idx_h], lse_ref[idx_b, idx_h])


def test_decode_multi_fault_injection_times_out_and_recovers(monkeypatch):
    # ATTN_FAULT_INJECT=skip_arrive: one softmax thread of CTA 0 withholds its P-ready arrival for the CTA's second
    # tile; the MMA warp's bounded wait runs out (about a second), the CTA winds down (copies and MMAs drained,
    # TMEM freed, its partials never published), the status word reports the timeout -- reading it re-zeroes the
    # row counters that the unpublished partials left behind -- and the next clean call is correct.
    B, Hq, Hkv, Lq, L = 4, 32, 8, 8, 8192  # ~14 tiles per CTA, so CTA 0 has a second tile
    q, kc, vc, _ = make_decode_multi(B, Hq, Hkv, Lq, L, 128, seed=1701)
    lens = torch.tensor([L, L - 300, 5000, 777], dtype=torch.int32)
    AB.attn_get_device_status()
    monkeypatch.setenv("ATTN_FAULT_INJECT", "skip_arrive")
    run(q, kc, vc, lens)
    assert AB.attn_get_device_status() == AB.ATTN_ERR_DEVICE_TIMEOUT
    monkeypatch.delenv("ATTN_FAULT_INJECT")
    O, lse = run(q, kc, vc, lens)
    assert AB.attn_get_device_status() == AB.ATTN_OK
    O_ref, lse_ref = oracle.decode_multi(q, kc, vc, lens.tolist(), 128 ** -0.5)
    assert_attn_close(O, lse, O_ref, lse_ref)
