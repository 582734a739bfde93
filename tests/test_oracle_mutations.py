"""Plant plausible mistakes in the oracle (on the CPU) and check the pins catch each.

Every mutation below swaps one helper of ``oracle.sdpa`` for a wrong version
-- a dropped term, a wrong sign or index, a transposed or swapped operand --
and runs the full pin list of ``test_oracle_pins.py``.  A mutation that no
pin notices would mean the pins do not fix that part of the oracle.
"""
import numpy as np
import pytest

from oracle import sdpa as OA
from tests.test_oracle_pins import PINS

_orig = {name: getattr(OA, name) for name in
         ("scores", "visible_mask", "kv_head_of", "softmax_two_pass", "log_sum_exp", "attention_head",
          "decode_multi", "rope_rotate", "_rope_q_k", "attention_varlen")}


def _varlen_keys_at_query_offsets(q, k, v, cu_seqlens_q, cu_seqlens_k, scale, causal, rope=None):
    # each packed sequence's keys sliced with the query offsets (right only while the two layouts coincide)
    return _orig["attention_varlen"](q, k, v, cu_seqlens_q, cu_seqlens_q, scale, causal, rope=rope)


def _rope_backwards(x, positions, cos, sin, style):
    return _orig["rope_rotate"](x, positions, cos, -np.asarray(sin), style)


def _rope_styles_swapped(x, positions, cos, sin, style):
    return _orig["rope_rotate"](x, positions, cos, sin, "interleaved" if style == "half" else "half")


def _rope_query_from_zero(Qh, Kh, Lq, Lkv, rope, rotate_k=True):
    # queries rotated to positions 0 .. Lq-1 instead of Lkv-Lq .. Lkv-1
    if rope is None:
        return Qh, Kh
    cos, sin, style = rope
    Qh = OA.rope_rotate(Qh, np.arange(Lq), cos, sin, style)
    if rotate_k:
        Kh = OA.rope_rotate(Kh, np.arange(Lkv), cos, sin, style)
    return Qh, Kh


def _rope_unrounded(Qh, Kh, Lq, Lkv, rope, rotate_k=True):
    if rope is None:
        return Qh, Kh
    cos, sin, style = rope
    Qh = OA.rope_rotate(Qh, np.arange(Lq) + (Lkv - Lq), cos, sin, style)
    if rotate_k:
        Kh = OA.rope_rotate(Kh, np.arange(Lkv), cos, sin, style)
    return Qh, Kh


def _rope_keys_not_rotated(Qh, Kh, Lq, Lkv, rope, rotate_k=True):
    return _orig["_rope_q_k"](Qh, Kh, Lq, Lkv, rope, rotate_k=False)


def _softmax_wrong_axis(S, visible):
    Sm = np.where(visible, S, -np.inf)
    m = np.max(Sm, axis=1, initial=-np.inf)
    E = np.where(visible, np.exp(Sm - np.where(np.isfinite(m), m, 0.0)[:, None]), 0.0)
    l = E.sum(axis=1)
    col = E.sum(axis=0, keepdims=True)
    return E / np.where(col > 0, col, 1.0), m, l


def _softmax_sign(S, visible):
    Sm = np.where(visible, S, -np.inf)
    m = np.max(Sm, axis=1, initial=-np.inf)
    ms = np.where(np.isfinite(m), m, 0.0)[:, None]
    E = np.where(visible, np.exp(np.where(visible, ms - S, 0.0)), 0.0)
    l = E.sum(axis=1)
    return E / np.where(l > 0, l, 1.0)[:, None], m, l


def _attention_head_k_for_v(Qh, Kh, Vh, scale, causal, visible=None):
    return _orig["attention_head"](Qh, Kh, Kh[:, : Vh.shape[1]] if Kh.shape[1] >= Vh.shape[1] else Vh,
                                   scale, causal, visible)


def _multi_with_mask(mask_of):
    """decode_multi with the visible set of token t over n keys given by mask_of(Lq, n) instead."""
    def bad(q, kcache, vcache, kv_lens, scale, heads=None, rope=None):
        q = OA.to_f64(q)
        B, Hq, Lq, D = q.shape
        Hkv = kcache.shape[1]
        O = np.full((B, Hq, Lq, vcache.shape[3]), np.nan)
        lse = np.full((B, Hq, Lq), np.nan)
        for b in range(B):
            n = int(kv_lens[b])
            for h in range(Hq):
                hk = OA.kv_head_of(h, Hq, Hkv)
                O[b, h], lse[b, h] = OA.attention_head(q[b, h], OA.to_f64(kcache[b, hk, :n]),
                                                       OA.to_f64(vcache[b, hk, :n]), scale, True,
                                                       visible=mask_of(Lq, n))
        return O, lse
    return bad


def _head_mask_before_scale(Qh, Kh, Vh, scale, causal, visible=None):
    # the mask applied to the raw scores, then the scale: right for scale > 0 only (-inf * 0 is NaN, and a
    # negative scale turns masked keys into +inf)
    Lq, Lkv = Qh.shape[0], Kh.shape[0]
    if visible is None:
        visible = OA.visible_mask(Lq, Lkv, causal)
    with np.errstate(invalid="ignore"):
        S = scale * np.where(visible, Qh @ Kh.T, -np.inf)
        P, m, l = OA.softmax_two_pass(S, np.ones_like(visible))
    return P @ Vh, OA.log_sum_exp(m, l)


def _scores_abs_scale(Qh, Kh, scale):
    return abs(scale) * (Qh @ Kh.T)


MUTATIONS = {
    "scale_dropped": ("scores", lambda Qh, Kh, scale: Qh @ Kh.T),
    "logit_sign": ("scores", lambda Qh, Kh, scale: -scale * (Qh @ Kh.T)),
    "mask_top_left": ("visible_mask", lambda Lq, Lkv, causal: (np.arange(Lkv)[None, :] <= np.arange(Lq)[:, None])
                      if causal else np.ones((Lq, Lkv), bool)),
    "mask_off_by_one": ("visible_mask", lambda Lq, Lkv, causal: (np.arange(Lkv)[None, :] < np.arange(Lq)[:, None]
                                                                + (Lkv - Lq)) if causal else np.ones((Lq, Lkv), bool)),
    "mask_ignored": ("visible_mask", lambda Lq, Lkv, causal: np.ones((Lq, Lkv), bool)),
    "gqa_modulo": ("kv_head_of", lambda hq, Hq, Hkv: hq % Hkv),
    "softmax_wrong_axis": ("softmax_two_pass", _softmax_wrong_axis),
    "softmax_exp_sign": ("softmax_two_pass", _softmax_sign),
    "lse_log2": ("log_sum_exp", lambda m, l: np.where(l > 0, m + np.log2(np.where(l > 0, l, 1.0)), -np.inf)),
    "lse_drops_max": ("log_sum_exp", lambda m, l: np.where(l > 0, np.log(np.where(l > 0, l, 1.0)), -np.inf)),
    "k_used_for_v": ("attention_head", _attention_head_k_for_v),
    "multi_sees_whole_cache": ("decode_multi", _multi_with_mask(lambda Lq, n: np.ones((Lq, n), bool))),
    "multi_top_left": ("decode_multi", _multi_with_mask(
        lambda Lq, n: np.arange(n)[None, :] <= np.arange(Lq)[:, None])),
    "multi_excludes_own_key": ("decode_multi", _multi_with_mask(
        lambda Lq, n: np.arange(n)[None, :] < np.arange(Lq)[:, None] + (n - Lq))),
    "rope_backwards": ("rope_rotate", _rope_backwards),
    "rope_styles_swapped": ("rope_rotate", _rope_styles_swapped),
    "rope_query_from_zero": ("_rope_q_k", _rope_query_from_zero),
    "rope_keys_not_rotated": ("_rope_q_k", _rope_keys_not_rotated),
    "rope_unrounded": ("_rope_q_k", _rope_unrounded),
    "varlen_keys_at_query_offsets": ("attention_varlen", _varlen_keys_at_query_offsets),
    "mask_before_scale": ("attention_head", _head_mask_before_scale),
    "scale_sign_dropped": ("scores", _scores_abs_scale),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_some_pin_catches(name, monkeypatch):
    attr, bad = MUTATIONS[name]
    monkeypatch.setattr(OA, attr, bad)
    caught = []
    for pin in PINS:
        try:
            pin()
        except Exception:  # an assertion or a shape error both mean the pin noticed
            caught.append(pin.__name__)
    assert caught, f"mutation {name} passed every pin"
