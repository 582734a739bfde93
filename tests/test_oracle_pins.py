"""Pins of the fp64 oracle against things other than itself (CPU only).

Each pin checks the oracle against a fact fixed by the mathematics or by the
pages' definition of attention (Operator Fusion, GPU learning diary day 24,
§3.4: S = QK^T/sqrt(d) + mask, P = softmax(S), O = PV):

* a brute-force pure-Python loop on tiny shapes (independent arithmetic);
* closed forms: identical keys, a dominant logit, the causal first row, a
  single key, V = 1 (softmax rows sum to one), hand-worked rational cases;
* special cases that reduce to library routines: torch's fp64
  scaled_dot_product_attention for square masks, scipy's softmax and
  logsumexp for one query;
* structural reductions: GQA == MHA with repeated K/V heads, decode ==
  last row of causal prefill, packed sequences == per-sequence dense,
  scale folded into q, key permutation invariance, each token of a
  multi-token decode step == single-token decode over its own prefix.

``PINS`` lists every pin; ``tests/test_oracle_mutations.py`` plants mistakes
in the oracle and checks that some pin fails for each.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import sdpa as OA
from oracle.brute import attention_loops

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")
GOLDEN_ROPE = os.path.join(os.path.dirname(__file__), "golden", "rope_hand_worked.json")


def _rng(seed):
    return np.random.default_rng(seed)


def _qkv(seed, B, Hq, Hkv, Lq, Lkv, D, Dv=None):
    r = _rng(seed)
    Dv = D if Dv is None else Dv
    return (r.standard_normal((B, Hq, Lq, D)), r.standard_normal((B, Hkv, Lkv, D)),
            r.standard_normal((B, Hkv, Lkv, Dv)))


# ----------------------------------------------------------------------------- pins

def pin_brute_force():
    """Vectorised oracle == literal loops, on shapes covering every mask case."""
    cases = [
        (1, 2, 2, 7, 7, 5, False),
        (1, 2, 2, 9, 9, 4, True),
        (2, 4, 2, 3, 11, 8, True),   # Lq < Lkv causal: bottom-right offset
        (1, 2, 1, 12, 6, 3, True),   # Lq > Lkv causal: first rows see nothing
        (1, 3, 3, 5, 6, 6, False),
        (1, 1, 1, 6, 6, 6, True),    # square D == L catches a transposed operand
    ]
    for n, (B, Hq, Hkv, Lq, Lkv, D, causal) in enumerate(cases):
        q, k, v = _qkv(10 + n, B, Hq, Hkv, Lq, Lkv, D)
        scale = 0.37 + 0.1 * n
        O, lse = OA.attention(q, k, v, scale, causal)
        Ob, lseb = attention_loops(q, k, v, scale, causal)
        np.testing.assert_allclose(O, np.array(Ob), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, np.array(lseb), rtol=0, atol=1e-12)


def pin_rows_sum_to_one():
    """softmax rows sum to 1, so V == 1 gives O == 1 on every row that sees a key."""
    for causal, (Lq, Lkv) in [(False, (9, 13)), (True, (13, 13)), (True, (5, 17))]:
        q, k, _ = _qkv(20, 1, 2, 2, Lq, Lkv, 6)
        S = OA.scores(q[0, 0], k[0, 0], 0.8)
        P, _, _ = OA.softmax_two_pass(S, OA.visible_mask(Lq, Lkv, causal))
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        assert (P >= 0).all()
        ones = np.ones((1, 2, Lkv, 3))
        O, _ = OA.attention(q, k, ones, 0.8, causal)
        np.testing.assert_allclose(O, 1.0, rtol=0, atol=1e-14)


def pin_identical_keys():
    """All keys equal c: O_i = mean of the visible V rows, lse_i = scale q_i.c + ln(n_visible)."""
    r = _rng(30)
    Lq, Lkv, D = 6, 10, 4
    c = r.standard_normal(D)
    q = r.standard_normal((1, 1, Lq, D))
    k = np.broadcast_to(c, (1, 1, Lkv, D)).copy()
    v = r.standard_normal((1, 1, Lkv, D))
    for causal in (False, True):
        O, lse = OA.attention(q, k, v, 0.5, causal)
        for i in range(Lq):
            n = (i + Lkv - Lq + 1) if causal else Lkv
            np.testing.assert_allclose(O[0, 0, i], v[0, 0, :n].mean(axis=0), atol=1e-13)
            assert abs(lse[0, 0, i] - (0.5 * q[0, 0, i] @ c + math.log(n))) < 1e-13


def pin_dominant_logit():
    """One key aligned with q and 50x longer dominates: O ~ V[k*], lse ~ its logit."""
    r = _rng(40)
    D, Lkv, kstar = 16, 12, 7
    q = r.standard_normal((1, 1, 1, D))
    k = 0.01 * r.standard_normal((1, 1, Lkv, D))
    k[0, 0, kstar] = 50.0 * q[0, 0, 0] / np.linalg.norm(q[0, 0, 0])
    v = r.standard_normal((1, 1, Lkv, D))
    O, lse = OA.attention(q, k, v, 1.0, False)
    logit = q[0, 0, 0] @ k[0, 0, kstar]
    assert logit > 40
    np.testing.assert_allclose(O[0, 0, 0], v[0, 0, kstar], atol=1e-9)
    assert abs(lse[0, 0, 0] - logit) < 1e-9


def pin_causal_first_row():
    """Square causal: row 0 sees only key 0, so O[0] = V[0] and lse[0] = S[0,0]."""
    q, k, v = _qkv(50, 2, 3, 3, 8, 8, 5)
    O, lse = OA.attention(q, k, v, 0.3, True)
    np.testing.assert_allclose(O[:, :, 0], v[:, :, 0], atol=1e-15)
    np.testing.assert_allclose(lse[:, :, 0], 0.3 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]), atol=1e-14)


def pin_single_key():
    """Lkv == 1: every row's weight is 1 on the only key."""
    q, k, v = _qkv(60, 1, 2, 2, 4, 1, 3)
    O, lse = OA.attention(q, k, v, 0.9, False)
    np.testing.assert_allclose(O, np.broadcast_to(v, O.shape), atol=1e-15)
    np.testing.assert_allclose(lse[0, 0], 0.9 * q[0, 0] @ k[0, 0, 0], atol=1e-14)


def pin_hand_worked_golden():
    """Cases worked by hand with rational softmax weights (tests/golden/hand_worked.json)."""
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        O, lse = OA.attention(np.array(c["q"]), np.array(c["k"]), np.array(c["v"]), c["scale"], c["causal"])
        np.testing.assert_allclose(O, np.array(c["O"]), rtol=0, atol=1e-14, err_msg=c["name"])
        np.testing.assert_allclose(lse, np.array(c["lse"]), rtol=0, atol=1e-14, err_msg=c["name"])


def pin_torch_sdpa():
    """torch's fp64 CPU scaled_dot_product_attention (library routine), where its
    causal convention (top-left) coincides with ours: square masks."""
    F = torch.nn.functional
    for B, Hq, Hkv, L, D, causal in [(2, 4, 4, 17, 8, False), (1, 4, 2, 23, 16, True), (1, 8, 2, 5, 4, False)]:
        q, k, v = _qkv(70 + L, B, Hq, Hkv, L, L, D)
        O, _ = OA.attention(q, k, v, 0.25, causal)
        tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
        ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=0.25, enable_gqa=(Hq != Hkv))
        np.testing.assert_allclose(O, ref.numpy(), atol=1e-12)


def pin_scipy_single_query():
    """One query: O = softmax(scale K q) V and lse = logsumexp(scale K q) (scipy routines)."""
    from scipy.special import logsumexp, softmax

    r = _rng(80)
    D, Lkv = 12, 31
    q = r.standard_normal((1, 1, 1, D))
    k = r.standard_normal((1, 1, Lkv, D))
    v = r.standard_normal((1, 1, Lkv, D))
    O, lse = OA.attention(q, k, v, 0.6, False)
    z = 0.6 * (k[0, 0] @ q[0, 0, 0])
    np.testing.assert_allclose(O[0, 0, 0], softmax(z) @ v[0, 0], atol=1e-13)
    assert abs(lse[0, 0, 0] - logsumexp(z)) < 1e-13


def pin_gqa_equals_mha():
    """Grouped heads == multi-head attention with each K/V head repeated over its query group."""
    B, Hq, Hkv, L, D = 2, 8, 2, 9, 4
    q, k, v = _qkv(90, B, Hq, Hkv, L, L + 3, D)
    g = Hq // Hkv
    for causal in (False, True):
        O, lse = OA.attention(q, k, v, 0.5, causal)
        Om, lsem = OA.attention(q, np.repeat(k, g, axis=1), np.repeat(v, g, axis=1), 0.5, causal)
        np.testing.assert_allclose(O, Om, atol=1e-14)
        np.testing.assert_allclose(lse, lsem, atol=1e-14)


def pin_decode_is_last_causal_row():
    """Decode over kv_len keys == the last row of causal prefill over those keys."""
    r = _rng(100)
    B, Hq, Hkv, Lmax, D = 3, 4, 2, 16, 8
    lens = [16, 5, 1]
    qd = r.standard_normal((B, Hq, D))
    kc = r.standard_normal((B, Hkv, Lmax, D))
    vc = r.standard_normal((B, Hkv, Lmax, D))
    O, lse = OA.decode(qd, kc, vc, lens, 0.4)
    for b, n in enumerate(lens):
        qp = r.standard_normal((1, Hq, n, D))
        qp[0, :, n - 1] = qd[b]
        Op, lsep = OA.attention(qp, kc[b:b + 1, :, :n], vc[b:b + 1, :, :n], 0.4, True)
        np.testing.assert_allclose(O[b], Op[0, :, n - 1], atol=1e-14)
        np.testing.assert_allclose(lse[b], lsep[0, :, n - 1], atol=1e-14)


def pin_scale_folds_into_q():
    """scale s with q == scale 1 with s*q (the scale multiplies the logits)."""
    q, k, v = _qkv(110, 1, 2, 2, 6, 9, 5)
    for causal in (False, True):
        O1, l1 = OA.attention(q, k, v, 0.3, causal)
        O2, l2 = OA.attention(0.3 * q, k, v, 1.0, causal)
        np.testing.assert_allclose(O1, O2, atol=1e-14)
        np.testing.assert_allclose(l1, l2, atol=1e-14)


def pin_key_permutation():
    """Non-causal: permuting K and V rows together leaves O and lse unchanged."""
    q, k, v = _qkv(120, 1, 2, 2, 5, 11, 4)
    perm = _rng(121).permutation(11)
    O1, l1 = OA.attention(q, k, v, 0.7, False)
    O2, l2 = OA.attention(q, k[:, :, perm], v[:, :, perm], 0.7, False)
    np.testing.assert_allclose(O1, O2, atol=1e-14)
    np.testing.assert_allclose(l1, l2, atol=1e-14)


def pin_varlen_is_per_sequence_dense():
    """Packed sequences == dense attention run on each sequence's own slices."""
    r = _rng(130)
    lens = [5, 1, 9, 3]
    cu = np.concatenate([[0], np.cumsum(lens)])
    Hq, Hkv, D = 4, 2, 6
    q = r.standard_normal((cu[-1], Hq, D))
    k = r.standard_normal((cu[-1], Hkv, D))
    v = r.standard_normal((cu[-1], Hkv, D))
    for causal in (False, True):
        O, lse = OA.attention_varlen(q, k, v, cu, cu, 0.5, causal)
        for s in range(len(lens)):
            sl = slice(cu[s], cu[s + 1])
            Od, lsed = OA.attention(q[sl].transpose(1, 0, 2)[None], k[sl].transpose(1, 0, 2)[None],
                                    v[sl].transpose(1, 0, 2)[None], 0.5, causal)
            np.testing.assert_allclose(O[sl], Od[0].transpose(1, 0, 2), atol=1e-14)
            np.testing.assert_allclose(lse[sl], lsed[0].T, atol=1e-14)
        Ob, lseb = attention_loops(q[:5].transpose(1, 0, 2)[None], k[:5].transpose(1, 0, 2)[None],
                                   v[:5].transpose(1, 0, 2)[None], 0.5, causal)
        np.testing.assert_allclose(O[:5], np.array(Ob)[0].transpose(1, 0, 2), atol=1e-12)


def pin_rows_equal_full():
    """Row-sampled helpers reproduce the corresponding rows of the full computation."""
    q, k, v = _qkv(140, 2, 4, 2, 10, 10, 4)
    O, lse = OA.attention(q, k, v, 0.5, True)
    rows = [0, 3, 9]
    Or, lr = OA.attention_rows(q, k, v, 0.5, True, 1, 3, rows)
    np.testing.assert_allclose(Or, O[1, 3, rows], atol=1e-15)
    np.testing.assert_allclose(lr, lse[1, 3, rows], atol=1e-15)
    r = _rng(141)
    lens = [4, 7]
    cu = np.array([0, 4, 11])
    qv, kv, vv = (r.standard_normal((11, 4, 4)), r.standard_normal((11, 2, 4)), r.standard_normal((11, 2, 4)))
    Ov, lv = OA.attention_varlen(qv, kv, vv, cu, cu, 0.5, True)
    Ovr, lvr = OA.attention_varlen_rows(qv, kv, vv, cu, cu, 0.5, True, 1, 2, [0, 6])
    np.testing.assert_allclose(Ovr, Ov[[4, 10], 2], atol=1e-15)
    np.testing.assert_allclose(lvr, lv[[4, 10], 2], atol=1e-15)


def pin_empty_rows():
    """Rows that see no key: O = 0 and lse = -inf (causal Lq > Lkv; decode kv_len == 0)."""
    q, k, v = _qkv(150, 1, 1, 1, 6, 3, 2)
    O, lse = OA.attention(q, k, v, 1.0, True)
    assert np.all(O[0, 0, :3] == 0) and np.all(np.isneginf(lse[0, 0, :3]))
    assert np.all(np.isfinite(lse[0, 0, 3:]))
    r = _rng(151)
    Od, lsed = OA.decode(r.standard_normal((2, 2, 4)), r.standard_normal((2, 1, 5, 4)),
                         r.standard_normal((2, 1, 5, 4)), [0, 5], 0.5)
    assert np.all(Od[0] == 0) and np.all(np.isneginf(lsed[0]))
    assert np.all(np.isfinite(lsed[1]))


def pin_bf16_inputs_promote_exactly():
    """bf16 torch inputs reach fp64 unchanged (every bf16 value is exact in fp64)."""
    t = torch.tensor([1.0 + 2 ** -7, -3.0, 2.0 ** -100], dtype=torch.bfloat16)
    np.testing.assert_array_equal(OA.to_f64(t), np.array([1.0 + 2 ** -7, -3.0, 2.0 ** -100]))


def pin_decode_multi_rows_are_single_decodes():
    """Token t of a multi-token decode step == single-token decode over the keys up to its own position
    (kv_len - Lq + t + 1 of them; none when that is <= 0)."""
    r = _rng(160)
    B, Hq, Hkv, Lq, Lmax, D = 3, 4, 2, 5, 12, 6
    lens = [12, 7, 3]  # the last sequence has kv_len < Lq: its first tokens see no key
    q = r.standard_normal((B, Hq, Lq, D))
    kc = r.standard_normal((B, Hkv, Lmax, D))
    vc = r.standard_normal((B, Hkv, Lmax, D))
    O, lse = OA.decode_multi(q, kc, vc, lens, 0.45)
    for t in range(Lq):
        lens_t = [max(0, n - Lq + t + 1) for n in lens]
        Od, lsed = OA.decode(q[:, :, t], kc, vc, lens_t, 0.45)
        np.testing.assert_allclose(O[:, :, t], Od, atol=1e-14, err_msg=f"token {t}")
        np.testing.assert_allclose(lse[:, :, t], lsed, atol=1e-14, err_msg=f"token {t}")
    assert np.all(O[2, :, :2] == 0) and np.all(np.isneginf(lse[2, :, :2]))


def pin_decode_multi_brute_force():
    """Multi-token decode == the literal loops (bottom-right causal) over each sequence's cache prefix."""
    r = _rng(161)
    B, Hq, Hkv, Lq, Lmax, D = 2, 4, 2, 3, 9, 4
    lens = [9, 4]
    q = r.standard_normal((B, Hq, Lq, D))
    kc = r.standard_normal((B, Hkv, Lmax, D))
    vc = r.standard_normal((B, Hkv, Lmax, D))
    O, lse = OA.decode_multi(q, kc, vc, lens, 0.7)
    for b, n in enumerate(lens):
        Ob, lb = attention_loops(q[b:b + 1], kc[b:b + 1, :, :n], vc[b:b + 1, :, :n], 0.7, True)
        np.testing.assert_allclose(O[b:b + 1], np.array(Ob), atol=1e-13)
        np.testing.assert_allclose(lse[b:b + 1], np.array(lb), atol=1e-13)


def pin_decode_multi_golden():
    """The hand-worked causal 2x2 case as a two-token step over a cache whose rows past kv_len are NaN."""
    with open(GOLDEN) as f:
        c = next(x for x in json.load(f)["cases"] if x["name"].startswith("causal 2x2"))
    q, k, v = np.array(c["q"]), np.array(c["k"]), np.array(c["v"])
    pad = np.full((1, 1, 3, 2), np.nan)
    kc, vc = np.concatenate([k, pad], axis=2), np.concatenate([v, pad], axis=2)
    O, lse = OA.decode_multi(q, kc, vc, [2], c["scale"])
    np.testing.assert_allclose(O, np.array(c["O"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, np.array(c["lse"]), rtol=0, atol=1e-14)


def _tables(max_pos, D, base=10000.0):
    ang = np.arange(max_pos)[:, None] * base ** (-np.arange(D // 2) * 2.0 / D)[None, :]
    return np.cos(ang), np.sin(ang)


def pin_rope_golden():
    """Rotations and one rotated attention worked by hand (tests/golden/rope_hand_worked.json)."""
    with open(GOLDEN_ROPE) as f:
        g = json.load(f)
    for c in g["rotate"]:
        out = OA.rope_rotate(np.array([c["x"]]), [0], np.array([c["cos"]]), np.array([c["sin"]]), c["style"])
        np.testing.assert_allclose(out[0], c["out"], rtol=0, atol=1e-15, err_msg=c["name"])
    for c in g["bf16_rounding"]:
        assert OA.round_bf16(np.array([c["x"]]))[0] == c["out"], c
    for c in g["attention"]:
        rope = (np.array(c["cos"]), np.array(c["sin"]), c["style"])
        O, lse = OA.attention(np.array(c["q"]), np.array(c["k"]), np.array(c["v"]), c["scale"], c["causal"], rope=rope)
        np.testing.assert_allclose(O, np.array(c["O"]), rtol=0, atol=1e-13, err_msg=c["name"])
        np.testing.assert_allclose(lse, np.array(c["lse"]), rtol=0, atol=1e-13, err_msg=c["name"])


def pin_round_bf16_matches_torch():
    """Rounding to bf16 agrees with torch's fp32 -> bf16 cast (library routine) on random and edge values."""
    r = _rng(176)
    x = np.concatenate([r.standard_normal(5000) * 10.0 ** r.integers(-6, 6, 5000), [0.0, -0.0, 65504.0, 1e-40]])
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(OA.round_bf16(x), want)


def pin_rope_complex_form():
    """Interleaved RoPE == multiplying each pair, read as a complex number, by cos + i sin (numpy complex)."""
    r = _rng(170)
    L, D = 7, 10
    x = r.standard_normal((L, D))
    cos, sin = _tables(20, D)
    pos = r.integers(0, 20, L)
    z = (x[:, 0::2] + 1j * x[:, 1::2]) * (cos[pos] + 1j * sin[pos])
    want = np.empty_like(x)
    want[:, 0::2], want[:, 1::2] = z.real, z.imag
    np.testing.assert_allclose(OA.rope_rotate(x, pos, cos, sin, "interleaved"), want, atol=1e-14)


def pin_rope_half_is_permuted_interleaved():
    """Half-split RoPE == interleaved RoPE on the dims reordered (0, D/2, 1, D/2+1, ...) and back."""
    r = _rng(171)
    L, D = 5, 8
    x = r.standard_normal((L, D))
    cos, sin = _tables(9, D)
    pos = r.integers(0, 9, L)
    perm = np.stack([np.arange(D // 2), np.arange(D // 2) + D // 2], axis=1).reshape(-1)
    got = OA.rope_rotate(x, pos, cos, sin, "half")
    via = np.empty_like(x)
    via[:, perm] = OA.rope_rotate(x[:, perm], pos, cos, sin, "interleaved")
    np.testing.assert_allclose(got, via, atol=1e-15)


def pin_rope_norms_and_relative_positions():
    """A rotation keeps every pair's length, and rotated dot products depend only on the position difference."""
    r = _rng(172)
    D = 16
    cos, sin = _tables(64, D)
    q, k = r.standard_normal((3, D)), r.standard_normal((3, D))
    for style in ("half", "interleaved"):
        rq = OA.rope_rotate(q, [5, 9, 30], cos, sin, style)
        np.testing.assert_allclose(np.linalg.norm(rq, axis=1), np.linalg.norm(q, axis=1), atol=1e-13)
        for s in (1, 17):
            a = OA.rope_rotate(q, [5, 9, 30], cos, sin, style) @ OA.rope_rotate(k, [2, 9, 12], cos, sin, style).T
            b = OA.rope_rotate(q, [5 + s, 9 + s, 30 + s], cos, sin, style) @ \
                OA.rope_rotate(k, [2 + s, 9 + s, 12 + s], cos, sin, style).T
            np.testing.assert_allclose(np.diag(a), np.diag(b), atol=1e-12)


def pin_rope_decode_is_last_prefill_row():
    """Decode with RoPE over a cache of rotated keys == the last row of rotated causal prefill."""
    r = _rng(173)
    B, Hq, Hkv, Lmax, D = 2, 4, 2, 12, 8
    lens = [12, 5]
    cos, sin = _tables(16, D)
    for style in ("half", "interleaved"):
        rope = (cos, sin, style)
        qd = r.standard_normal((B, Hq, D))
        k = r.standard_normal((B, Hkv, Lmax, D))
        v = r.standard_normal((B, Hkv, Lmax, D))
        kc = OA.round_bf16(OA.rope_rotate(k, np.arange(Lmax), cos, sin, style))  # the cache holds bf16 rotated keys
        O, lse = OA.decode(qd, kc, v, lens, 0.4, rope=rope)
        Om, lsem = OA.decode_multi(qd[:, :, None], kc, v, lens, 0.4, rope=rope)
        for b, n in enumerate(lens):
            qp = r.standard_normal((1, Hq, n, D))
            qp[0, :, n - 1] = qd[b]
            Op, lsep = OA.attention(qp, k[b:b + 1, :, :n], v[b:b + 1, :, :n], 0.4, True, rope=rope)
            np.testing.assert_allclose(O[b], Op[0, :, n - 1], atol=1e-13)
            np.testing.assert_allclose(lse[b], lsep[0, :, n - 1], atol=1e-13)
            np.testing.assert_allclose(Om[b, :, 0], Op[0, :, n - 1], atol=1e-13)


def pin_rope_multi_tokens_are_prefill_rows():
    """Multi-token decode with RoPE == the last Lq rows of rotated causal prefill over each sequence's keys."""
    r = _rng(174)
    B, Hq, Hkv, Lq, Lmax, D = 2, 4, 2, 3, 10, 8
    lens = [10, 6]
    cos, sin = _tables(12, D)
    rope = (cos, sin, "half")
    q = r.standard_normal((B, Hq, Lq, D))
    k = r.standard_normal((B, Hkv, Lmax, D))
    v = r.standard_normal((B, Hkv, Lmax, D))
    kc = OA.round_bf16(OA.rope_rotate(k, np.arange(Lmax), cos, sin, "half"))
    O, lse = OA.decode_multi(q, kc, v, lens, 0.6, rope=rope)
    for b, n in enumerate(lens):
        Op, lsep = OA.attention(q[b:b + 1], k[b:b + 1, :, :n], v[b:b + 1, :, :n], 0.6, True, rope=rope)
        np.testing.assert_allclose(O[b], Op[0], atol=1e-13)
        np.testing.assert_allclose(lse[b], lsep[0], atol=1e-13)


def pin_rope_rows_and_varlen_agree_with_dense():
    """The row-sampled and packed forms rotate with the same positions as dense prefill, also when a packed
    sequence has fewer queries than keys."""
    r = _rng(175)
    Hq, Hkv, D = 4, 2, 8
    cos, sin = _tables(32, D)
    rope = (cos, sin, "interleaved")
    lens = [9, 14]
    cu = [0, 9, 23]
    q, k, v = r.standard_normal((23, Hq, D)), r.standard_normal((23, Hkv, D)), r.standard_normal((23, Hkv, D))
    Ov, lv = OA.attention_varlen(q, k, v, cu, cu, 0.5, True, rope=rope)
    for s, n in enumerate(lens):
        a, e = cu[s], cu[s + 1]
        qd, kd, vd = (x[a:e].transpose(1, 0, 2)[None] for x in (q, k, v))
        Od, ld = OA.attention(qd, kd, vd, 0.5, True, rope=rope)
        np.testing.assert_allclose(Ov[a:e].transpose(1, 0, 2), Od[0], atol=1e-13)
        rows = np.array([0, n - 1, n // 2])
        Orr, lrr = OA.attention_rows(qd, kd, vd, 0.5, True, 0, 3, rows, rope=rope)
        np.testing.assert_allclose(Orr, Od[0, 3, rows], atol=1e-13)
        Ovr, lvr = OA.attention_varlen_rows(q, k, v, cu, cu, 0.5, True, s, 3, rows, rope=rope)
        np.testing.assert_allclose(Ovr, Od[0, 3, rows], atol=1e-13)
    # fewer queries than keys in each sequence: the packed forms place sequence s's queries at Lkv_s - Lq_s + i
    # of that sequence alone, as dense prefill does for the same slices
    q_lens, k_lens = [4, 11], [9, 14]
    cq, ck = [0, 4, 15], [0, 9, 23]
    q = r.standard_normal((15, Hq, D))
    Ov, lv = OA.attention_varlen(q, k, v, cq, ck, 0.5, True, rope=rope)
    for s in range(2):
        qd = q[cq[s]:cq[s + 1]].transpose(1, 0, 2)[None]
        kd, vd = (x[ck[s]:ck[s + 1]].transpose(1, 0, 2)[None] for x in (k, v))
        Od, ld = OA.attention(qd, kd, vd, 0.5, True, rope=rope)
        np.testing.assert_allclose(Ov[cq[s]:cq[s + 1]].transpose(1, 0, 2), Od[0], atol=1e-13)
        np.testing.assert_allclose(lv[cq[s]:cq[s + 1]].T, ld[0], atol=1e-13)
        rows = np.array([0, q_lens[s] - 1])
        Ovr, lvr = OA.attention_varlen_rows(q, k, v, cq, ck, 0.5, True, s, 1, rows, rope=rope)
        np.testing.assert_allclose(Ovr, Od[0, 1, rows], atol=1e-13)


def pin_scale_zero_is_uniform_average():
    """scale 0: every visible logit is 0, so O is the plain mean of the visible V rows and lse = ln(count).

    A closed form that needs no exponential: it pins where the scale is applied (before the mask is added --
    a mask applied to raw scores and then multiplied by 0 would give NaN) and the count of visible keys under
    the bottom-right causal alignment, for square, Lq < Lkv, Lq > Lkv (empty first rows), decode and multi-token
    decode alike."""
    for n, (Lq, Lkv, causal) in enumerate([(7, 7, True), (4, 9, True), (9, 5, True), (6, 8, False)]):
        q, k, v = _qkv(700 + n, 1, 4, 2, Lq, Lkv, 5)
        O, lse = OA.attention(q, k, v, 0.0, causal)
        for h in range(4):
            hk = h // 2
            for i in range(Lq):
                cnt = min(Lkv, i + (Lkv - Lq) + 1) if causal else Lkv
                if cnt <= 0:
                    assert lse[0, h, i] == -np.inf and not O[0, h, i].any()
                    continue
                np.testing.assert_allclose(O[0, h, i], v[0, hk, :cnt].mean(axis=0), atol=1e-14)
                assert abs(lse[0, h, i] - math.log(cnt)) < 1e-14
    r = _rng(710)
    qd, kc, vc = r.standard_normal((2, 4, 6)), r.standard_normal((2, 2, 12, 6)), r.standard_normal((2, 2, 12, 6))
    lens = [12, 5]
    Od, ld = OA.decode(qd, kc, vc, lens, 0.0)
    qm = r.standard_normal((2, 4, 3, 6))
    Om, lm = OA.decode_multi(qm, kc, vc, lens, 0.0)
    for b, nb in enumerate(lens):
        for h in range(4):
            np.testing.assert_allclose(Od[b, h], vc[b, h // 2, :nb].mean(axis=0), atol=1e-14)
            assert abs(ld[b, h] - math.log(nb)) < 1e-14
            for t in range(3):
                cnt = nb - 3 + t + 1
                np.testing.assert_allclose(Om[b, h, t], vc[b, h // 2, :cnt].mean(axis=0), atol=1e-14)
                assert abs(lm[b, h, t] - math.log(cnt)) < 1e-14


def pin_negative_scale():
    """A negative scale against the literal loops, and scale -s with q equal to scale s with -q."""
    for n, (Lq, Lkv, causal) in enumerate([(6, 6, True), (3, 8, True), (5, 7, False)]):
        q, k, v = _qkv(720 + n, 1, 2, 1, Lq, Lkv, 4)
        O, lse = OA.attention(q, k, v, -0.61, causal)
        Ob, lseb = attention_loops(q, k, v, -0.61, causal)
        np.testing.assert_allclose(O, np.array(Ob), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, np.array(lseb), rtol=0, atol=1e-12)
        O2, l2 = OA.attention(-q, k, v, 0.61, causal)
        np.testing.assert_allclose(O, O2, atol=1e-14)
        np.testing.assert_allclose(lse, l2, atol=1e-14)
    # decode: the smallest logit now dominates -- the key most aligned with q gets the least weight
    r = _rng(730)
    qd = r.standard_normal((1, 1, 4))
    kc = np.zeros((1, 1, 3, 4))
    kc[0, 0, 0] = 40 * qd[0, 0] / np.linalg.norm(qd[0, 0])  # aligned with q: largest raw score
    kc[0, 0, 1] = -40 * qd[0, 0] / np.linalg.norm(qd[0, 0])  # opposite: smallest raw score
    vc = r.standard_normal((1, 1, 3, 4))
    O, _ = OA.decode(qd, kc, vc, [3], -1.0)
    np.testing.assert_allclose(O[0, 0], vc[0, 0, 1], atol=1e-12)


PINS = [
    pin_brute_force,
    pin_rows_sum_to_one,
    pin_identical_keys,
    pin_dominant_logit,
    pin_causal_first_row,
    pin_single_key,
    pin_hand_worked_golden,
    pin_torch_sdpa,
    pin_scipy_single_query,
    pin_gqa_equals_mha,
    pin_decode_is_last_causal_row,
    pin_scale_folds_into_q,
    pin_key_permutation,
    pin_varlen_is_per_sequence_dense,
    pin_rows_equal_full,
    pin_empty_rows,
    pin_bf16_inputs_promote_exactly,
    pin_decode_multi_rows_are_single_decodes,
    pin_decode_multi_brute_force,
    pin_decode_multi_golden,
    pin_rope_golden,
    pin_round_bf16_matches_torch,
    pin_rope_complex_form,
    pin_rope_half_is_permuted_interleaved,
    pin_rope_norms_and_relative_positions,
    pin_rope_decode_is_last_prefill_row,
    pin_rope_multi_tokens_are_prefill_rows,
    pin_rope_rows_and_varlen_agree_with_dense,
    pin_scale_zero_is_uniform_average,
    pin_negative_scale,
]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


def test_package_exports_match_module():
    assert oracle.attention is OA.attention and oracle.decode is OA.decode
