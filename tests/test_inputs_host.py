"""The seeded input generators (attention_attn_fwd_06_gb300/inputs.py) that both the oracle tests and the GPU
parity tests draw from: every parity claim rests on both sides seeing the same tensors, so the generators must be
deterministic for a seed, differ across seeds, and produce the shapes, dtypes and value structure their
workloads state (bf16 from N(0,1), lengths in range, packed offsets consistent)."""
import torch

from attention_attn_fwd_06_gb300.inputs import (WORKLOADS, make_decode, make_decode_multi, make_pages,
                                                make_prefill, make_varlen, rope_tables)


def test_generators_are_deterministic_per_seed():
    for make in (lambda s: make_prefill(2, 4, 2, 70, 90, 64, seed=s),
                 lambda s: make_decode(3, 8, 2, 100, 128, seed=s, kv_range=(1, 100)),
                 lambda s: make_decode_multi(2, 8, 2, 3, 50, 64, seed=s),
                 lambda s: make_varlen(3, 4, 2, 64, s, seq_range=(5, 40))):
        a, b, c = make(11), make(11), make(12)
        assert all(torch.equal(x, y) for x, y in zip(a, b))
        assert not all(torch.equal(x, y) for x, y in zip(a, c))


def test_prefill_shapes_dtypes_and_values():
    q, k, v = make_prefill(2, 8, 2, 33, 65, 128, seed=5)
    assert q.shape == (2, 8, 33, 128) and k.shape == (2, 2, 65, 128) and v.shape == k.shape
    assert q.dtype == k.dtype == v.dtype == torch.bfloat16
    x = torch.cat([q.float().flatten(), k.float().flatten(), v.float().flatten()])
    assert abs(x.mean().item()) < 0.05 and abs(x.std().item() - 1.0) < 0.05  # N(0,1) rounded to bf16


def test_decode_lengths_in_range():
    q, kc, vc, lens = make_decode(64, 4, 4, 300, 64, seed=6, kv_range=(17, 300))
    assert lens.dtype == torch.int32 and lens.shape == (64,)
    assert int(lens.min()) >= 17 and int(lens.max()) <= 300
    assert kc.shape == (64, 4, 300, 64)


def test_varlen_offsets_consistent():
    q, k, v, cu = make_varlen(5, 4, 2, 64, 9, seq_range=(3, 50))
    assert cu.dtype == torch.int32 and int(cu[0]) == 0 and bool((cu[1:] >= cu[:-1]).all())
    lens = (cu[1:] - cu[:-1])
    assert int(lens.min()) >= 3 and int(lens.max()) <= 50
    assert q.shape[0] == int(cu[-1]) == k.shape[0] == v.shape[0]


def test_pages_hold_the_cache_and_poison_the_rest():
    _, kc, vc, _ = make_decode(2, 2, 2, 40, 64, seed=3)
    kp, vp, table = make_pages(kc, vc, 16, seed=4)
    assert len(set(table.flatten().tolist())) == table.numel()  # no page shared
    for b in range(2):
        for i in range(table.shape[1]):
            lo, hi = 16 * i, min(40, 16 * (i + 1))
            assert torch.equal(kp[table[b, i], :, : hi - lo], kc[b, :, lo:hi])
            assert torch.equal(vp[table[b, i], :, : hi - lo], vc[b, :, lo:hi])
    used = set(table.flatten().tolist())
    spare = [p for p in range(kp.shape[0]) if p not in used]
    assert spare and all(torch.isnan(kp[p].float()).all() for p in spare)


def test_rope_tables_are_the_frequency_ladder():
    cos, sin = rope_tables(10, 8)
    assert cos.shape == sin.shape == (10, 4) and cos.dtype == torch.float32
    assert torch.allclose(cos * cos + sin * sin, torch.ones_like(cos), atol=1e-6)
    assert torch.allclose(cos[0], torch.ones(4)) and torch.allclose(sin[0], torch.zeros(4))
    # position 1, pair 0: angle 1 (base^0)
    assert abs(cos[1, 0].item() - 0.5403023) < 1e-6 and abs(sin[1, 0].item() - 0.8414710) < 1e-6


def test_workload_table_matches_the_stated_configs():
    w = WORKLOADS["decode_gqa"]
    assert (w.B, w.Hq, w.Hkv, w.D, w.L, tuple(w.kv_range)) == (8, 32, 8, 128, 4096, (512, 4096))
    w = WORKLOADS["decode_long"]
    assert (w.B, w.Hq, w.Hkv, w.D, tuple(w.kv_lens)) == (4, 32, 8, 128, (32768, 65536, 98304, 131072))
    w = WORKLOADS["prefill_causal"]
    assert (w.B, w.Hq, w.Hkv, w.D, w.L, w.causal) == (4, 32, 32, 128, 4096, True)
    w = WORKLOADS["prefill_noncausal_d64"]
    assert (w.B, w.Hq, w.Hkv, w.D, w.L, w.causal) == (2, 16, 16, 64, 8192, False)
    w = WORKLOADS["tiny_causal"]
    assert (w.B, w.Hq, w.Hkv, w.D, w.L, w.causal) == (1, 2, 2, 64, 128, True)
