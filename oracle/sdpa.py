"""Plain, slow, fp64 CPU oracle for scaled-dot-product attention forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It shares no code with the CUDA library.

What it computes is the unfused definition of attention as written in
"GPU 学习日报 Day 24：Operator Fusion" (Operator Fusion, GPU learning diary day 24),
§3.4 "Attention Fusion: FlashAttention", first listing (the standard chain):

    S = Q @ K^T,   S = S / sqrt(d) + mask,   P = softmax(S),   O = P @ V

with the softmax taken in two passes (a max reduction, then exponentiation and
normalisation), the way "Оптимизация Decoder Attention для LLM на GPU"
(Optimizing Decoder Attention for LLMs on GPU), section "Узкие места
традиционных подходов" (bottlenecks of traditional approaches), item 3,
describes the separate softmax kernel.  The same §3.4 states that the fused,
tiled, online-softmax kernel reaches this result up to floating-point rounding
(FAQ Q1 of the same page), so the plain definition is the oracle.

Readings taken where the pages leave a step open (each one is listed in the
design notes of the repository):

* ``scale`` multiplies the logits before the softmax (the §3.4 chain divides
  by sqrt(d); callers pass 1/sqrt(D) for that).
* The "+ mask" of §3.4 is the causal mask, aligned to the bottom-right corner:
  key j is visible to query i iff ``j <= i + (Lkv - Lq)``.  For Lq == Lkv this
  is the usual lower triangle; for single-token decode (Lq == 1) every cached
  key is visible, matching the decoder page's statement that each new token
  depends on all earlier tokens.
* Grouped-query heads use contiguous groups: query head ``hq`` reads key/value
  head ``hq // (Hq // Hkv)``.
* The per-row log-sum-exp is ``lse = m + ln(l)`` in natural log over the
  scaled (and masked) logits, with m the row max and l the row sum of
  ``exp(S - m)`` -- the two quantities the §3.4 online listing carries.
* A row with no visible key (only possible for causal Lq > Lkv, or a decode
  sequence with kv_len == 0) yields O = 0 and lse = -inf.
* RoPE (rotary position embedding), which "Что такое kernel fusion и как он
  применяется в LLM serving?" §3.5 and the Operator Fusion page's exercise 1
  name as fusable into the attention kernel without giving its formula, is
  read as the standard rotary embedding: pair i of a row at position p is
  turned by the angle whose cosine and sine the caller's tables hold at
  [p, i], ``(a, b) -> (a cos - b sin, b cos + a sin)``, the pairs being
  dims (i, i + D/2) ("half") or (2i, 2i + 1) ("interleaved").  Queries and
  keys take the positions the causal alignment gives them: key j sits at j,
  query i of Lq at ``Lkv - Lq + i``; a decode token at ``kv_len - Lq + t``.
  Cached keys are stored already rotated (decode rotates only q).  The
  rotated q and k are rounded to bf16 (nearest, ties to even) before the
  attention chain uses them: Operator Fusion's exercise 1 lists RoPE and
  attention as two ops of the unfused chain, and the tensor between them is
  held in the inputs' bf16, so that is the result a fused kernel reproduces.

Inputs are taken as given (typically bf16 values already rounded, passed as
float32/float64 arrays or CPU torch tensors) and promoted to fp64.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "to_f64",
    "kv_head_of",
    "visible_mask",
    "scores",
    "softmax_two_pass",
    "log_sum_exp",
    "attention_head",
    "attention",
    "attention_rows",
    "attention_varlen",
    "attention_varlen_rows",
    "decode",
    "decode_multi",
    "rope_rotate",
    "round_bf16",
]


def to_f64(x) -> np.ndarray:
    """Promote a numpy array or CPU torch tensor (any float dtype) to fp64 numpy."""
    if hasattr(x, "detach"):  # torch tensor; bf16 has no numpy dtype, go via fp32 (exact)
        x = x.detach().to("cpu")
        if str(x.dtype) in ("torch.bfloat16", "torch.float16"):
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def kv_head_of(hq: int, Hq: int, Hkv: int) -> int:
    """Key/value head read by query head ``hq`` (contiguous query-head groups)."""
    return hq // (Hq // Hkv)


def visible_mask(Lq: int, Lkv: int, causal: bool) -> np.ndarray:
    """Boolean [Lq, Lkv] matrix: True where key j is visible to query i.

    The "+ mask" term of the standard attention chain (Operator Fusion §3.4),
    read as a causal mask aligned to the bottom-right corner.
    """
    if not causal:
        return np.ones((Lq, Lkv), dtype=bool)
    i = np.arange(Lq)[:, None]
    j = np.arange(Lkv)[None, :]
    return j <= i + (Lkv - Lq)


def scores(Qh: np.ndarray, Kh: np.ndarray, scale: float) -> np.ndarray:
    """S = scale * Q K^T, materialised in full (Operator Fusion §3.4, first two lines)."""
    return scale * (Qh @ Kh.T)


def softmax_two_pass(S: np.ndarray, visible: np.ndarray):
    """Two-pass row softmax of the masked logits.

    Pass 1 reduces each row to its maximum m over the visible entries; pass 2
    exponentiates ``S - m``, sums to l and normalises (decoder-attention page,
    "bottlenecks of traditional approaches", item 3).  Returns (P, m, l); rows
    with nothing visible get P = 0, m = -inf, l = 0.
    """
    Sm = np.where(visible, S, -np.inf)
    m = np.max(Sm, axis=1, initial=-np.inf)  # pass 1
    has_key = np.isfinite(m)
    m_safe = np.where(has_key, m, 0.0)
    E = np.where(visible, np.exp(Sm - m_safe[:, None]), 0.0)  # pass 2
    l = E.sum(axis=1)
    P = np.where(has_key[:, None], E / np.where(has_key, l, 1.0)[:, None], 0.0)
    return P, m, l


def attention_head(Qh, Kh, Vh, scale: float, causal: bool, visible=None):
    """One (batch, head): O = softmax(scale Q K^T + mask) V and its row log-sum-exp.

    Qh [Lq, D], Kh [Lkv, D], Vh [Lkv, Dv] in fp64.  Returns O [Lq, Dv], lse [Lq].
    """
    Lq, Lkv = Qh.shape[0], Kh.shape[0]
    if visible is None:
        visible = visible_mask(Lq, Lkv, causal)
    S = scores(Qh, Kh, scale)
    P, m, l = softmax_two_pass(S, visible)
    O = P @ Vh
    return O, log_sum_exp(m, l)


def log_sum_exp(m: np.ndarray, l: np.ndarray) -> np.ndarray:
    """lse = m + ln(l): the natural-log normaliser of each softmax row; -inf where l == 0."""
    with np.errstate(divide="ignore"):
        return np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)


def rope_rotate(x, positions, cos, sin, style: str) -> np.ndarray:
    """Rotary position embedding of the rows of ``x`` (fp64).

    x [..., L, D]; positions [L] (row r sits at positions[r]); cos/sin
    [max_pos, D/2] tables whose row p holds the cosines and sines of the
    angles of the D/2 pairs at position p.  Pair i of a row, (a, b), becomes
    ``(a cos - b sin, b cos + a sin)`` -- a plane rotation of the pair.  Pairs
    are dims (i, i + D/2) for ``style == "half"`` and (2i, 2i + 1) for
    ``style == "interleaved"``.
    """
    x = to_f64(x)
    D = x.shape[-1]
    pos = np.asarray(positions, dtype=np.int64)
    c = to_f64(cos)[pos]  # [L, D/2]
    s = to_f64(sin)[pos]
    if style == "half":
        a, b = x[..., : D // 2], x[..., D // 2:]
        return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)
    if style == "interleaved":
        a, b = x[..., 0::2], x[..., 1::2]
        out = np.empty_like(x)
        out[..., 0::2] = a * c - b * s
        out[..., 1::2] = b * c + a * s
        return out
    raise ValueError(f"unknown rope style {style!r}")


def round_bf16(x) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (ties to even), returned as fp64.

    bf16 keeps the top 16 bits of an fp32 word; the value is first rounded to
    fp32 (exact for every value that is then representable in bf16), then its
    low 16 bits are rounded away with ties going to the even neighbour.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    finite = np.isfinite(f)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    out = np.where(finite, r, u).astype(np.uint32).view(np.float32)
    return out.astype(np.float64)


def _rope_q_k(Qh, Kh, Lq, Lkv, rope, rotate_k=True):
    """Rotate a head's query rows (positions Lkv - Lq + i) and key rows (positions j) when ``rope`` is given,
    rounding the rotated values to bf16 (the dtype of the tensor between RoPE and attention)."""
    if rope is None:
        return Qh, Kh
    cos, sin, style = rope
    Qh = round_bf16(rope_rotate(Qh, np.arange(Lq) + (Lkv - Lq), cos, sin, style))
    if rotate_k:
        Kh = round_bf16(rope_rotate(Kh, np.arange(Lkv), cos, sin, style))
    return Qh, Kh


def _check_heads(Hq: int, Hkv: int):
    if Hkv <= 0 or Hq % Hkv != 0:
        raise ValueError(f"Hq={Hq} must be a positive multiple of Hkv={Hkv}")


def attention(q, k, v, scale: float, causal: bool, rope=None):
    """Dense prefill: q [B,Hq,Lq,D], k/v [B,Hkv,Lkv,D] -> O [B,Hq,Lq,D], lse [B,Hq,Lq].

    ``rope = (cos, sin, style)`` rotates q and k first (see :func:`rope_rotate`).
    """
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    B, Hq, Lq, D = q.shape
    Hkv, Lkv = k.shape[1], k.shape[2]
    _check_heads(Hq, Hkv)
    O = np.zeros((B, Hq, Lq, v.shape[3]))
    lse = np.zeros((B, Hq, Lq))
    for b in range(B):
        for h in range(Hq):
            hk = kv_head_of(h, Hq, Hkv)
            Qh, Kh = _rope_q_k(q[b, h], k[b, hk], Lq, Lkv, rope)
            O[b, h], lse[b, h] = attention_head(Qh, Kh, v[b, hk], scale, causal)
    return O, lse


def attention_rows(q, k, v, scale: float, causal: bool, b: int, h: int, rows, rope=None):
    """Selected query rows of one (batch, head) of :func:`attention`.

    Each row is computed from its own definition (its scores against every
    key, its mask row, its two-pass softmax), so checking a sample of rows of a
    large problem costs O(rows * Lkv * D).
    """
    Hq, Lq = q.shape[1], q.shape[2]
    Hkv, Lkv = k.shape[1], k.shape[2]
    _check_heads(Hq, Hkv)
    rows = np.asarray(rows, dtype=np.int64)
    hk = kv_head_of(h, Hq, Hkv)
    vis = visible_mask(Lq, Lkv, causal)[rows]
    Qh = to_f64(q[b, h])[rows]  # promote only the slices this row set reads
    Kh = to_f64(k[b, hk])
    if rope is not None:
        cos, sin, style = rope
        Qh = round_bf16(rope_rotate(Qh, rows + (Lkv - Lq), cos, sin, style))
        Kh = round_bf16(rope_rotate(Kh, np.arange(Lkv), cos, sin, style))
    return attention_head(Qh, Kh, to_f64(v[b, hk]), scale, causal, visible=vis)


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool, rope=None):
    """Packed variable-length prefill.

    q [total_q, Hq, D], k/v [total_k, Hkv, D]; sequence s owns rows
    ``cu_seqlens_*[s] : cu_seqlens_*[s+1]``.  Each sequence is an independent
    attention problem with the bottom-right causal alignment of its own
    lengths.  Returns O [total_q, Hq, D], lse [total_q, Hq].
    """
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    cq = np.asarray(cu_seqlens_q, dtype=np.int64)
    ck = np.asarray(cu_seqlens_k, dtype=np.int64)
    Hq, Hkv = q.shape[1], k.shape[1]
    _check_heads(Hq, Hkv)
    O = np.zeros((q.shape[0], Hq, v.shape[2]))
    lse = np.full((q.shape[0], Hq), -np.inf)
    for s in range(len(cq) - 1):
        qs, qe, ks, ke = cq[s], cq[s + 1], ck[s], ck[s + 1]
        for h in range(Hq):
            hk = kv_head_of(h, Hq, Hkv)
            Qh, Kh = _rope_q_k(q[qs:qe, h], k[ks:ke, hk], qe - qs, ke - ks, rope)
            o, ls = attention_head(Qh, Kh, v[ks:ke, hk], scale, causal)
            O[qs:qe, h] = o
            lse[qs:qe, h] = ls
    return O, lse


def attention_varlen_rows(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool,
                          seq: int, h: int, rows, rope=None):
    """Selected rows (relative to the start of sequence ``seq``) of :func:`attention_varlen`."""
    cq = np.asarray(cu_seqlens_q, dtype=np.int64)
    ck = np.asarray(cu_seqlens_k, dtype=np.int64)
    Hq, Hkv = q.shape[1], k.shape[1]
    _check_heads(Hq, Hkv)
    rows = np.asarray(rows, dtype=np.int64)
    qs, qe, ks, ke = (int(x) for x in (cq[seq], cq[seq + 1], ck[seq], ck[seq + 1]))
    hk = kv_head_of(h, Hq, Hkv)
    vis = visible_mask(qe - qs, ke - ks, causal)[rows]
    Qh = to_f64(q[qs:qe, h])[rows]
    Kh = to_f64(k[ks:ke, hk])
    if rope is not None:
        cos, sin, style = rope
        Qh = round_bf16(rope_rotate(Qh, rows + ((ke - ks) - (qe - qs)), cos, sin, style))
        Kh = round_bf16(rope_rotate(Kh, np.arange(ke - ks), cos, sin, style))
    return attention_head(Qh, Kh, to_f64(v[ks:ke, hk]), scale, causal, visible=vis)


def decode(q, kcache, vcache, kv_lens, scale: float, heads=None, rope=None):
    """Single-token decode over a KV cache.

    q [B,Hq,D], kcache/vcache [B,Hkv,Lmax,D], kv_lens [B].  The new token of
    sequence b attends to cached keys ``0 .. kv_lens[b]-1`` (decoder-attention
    page, "structure of attention in decoding mode").  Returns O [B,Hq,D] and
    lse [B,Hq].  ``heads`` optionally restricts the work to a list of (b, hq)
    pairs; the other entries are left as NaN.  With ``rope = (cos, sin,
    style)`` the query is rotated to its position kv_lens[b] - 1; the cached
    keys are used as stored (already rotated).
    """
    q = to_f64(q)
    lens = np.asarray(kv_lens, dtype=np.int64)
    B, Hq, D = q.shape
    Hkv = kcache.shape[1]
    _check_heads(Hq, Hkv)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(Hq)]
    O = np.full((B, Hq, vcache.shape[3]), np.nan)
    lse = np.full((B, Hq), np.nan)
    for b, h in heads:
        n = int(lens[b])
        hk = kv_head_of(h, Hq, Hkv)
        # promote only the cache rows this sequence attends to
        Qh, _ = _rope_q_k(q[b, h][None, :], None, 1, n, rope, rotate_k=False)
        o, ls = attention_head(Qh, to_f64(kcache[b, hk, :n]), to_f64(vcache[b, hk, :n]), scale, causal=False)
        O[b, h], lse[b, h] = o[0], ls[0]
    return O, lse


def decode_multi(q, kcache, vcache, kv_lens, scale: float, heads=None, rope=None):
    """Decode of several new tokens per sequence over a KV cache.

    q [B,Hq,Lq,D], kcache/vcache [B,Hkv,Lmax,D], kv_lens [B].  Rows
    ``0 .. kv_lens[b]-1`` of sequence b's cache hold all of its keys, the Lq new
    tokens' own keys being the last Lq of them, so new token t (0-based) sits
    at position ``kv_lens[b] - Lq + t`` and attends to keys
    ``0 .. kv_lens[b] - Lq + t``: the causal mask of the Lq x kv_len score
    block aligned to its bottom-right corner, as for prefill.  The
    decoder-attention page ("Техника выжимания производительности", item 1,
    token-level parallelism) processes several query tokens of a step at once
    against K/V blocks loaded once; what each token computes is the single
    decode above over its own visible prefix.  Returns O [B,Hq,Lq,D] and
    lse [B,Hq,Lq]; ``heads`` optionally restricts the work to (b, hq) pairs,
    the other entries being NaN.  With ``rope = (cos, sin, style)`` token t
    is rotated to its position kv_lens[b] - Lq + t; cached keys are used as
    stored (already rotated).
    """
    q = to_f64(q)
    lens = np.asarray(kv_lens, dtype=np.int64)
    B, Hq, Lq, D = q.shape
    Hkv = kcache.shape[1]
    _check_heads(Hq, Hkv)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(Hq)]
    O = np.full((B, Hq, Lq, vcache.shape[3]), np.nan)
    lse = np.full((B, Hq, Lq), np.nan)
    for b, h in heads:
        n = int(lens[b])
        hk = kv_head_of(h, Hq, Hkv)
        Qh, _ = _rope_q_k(q[b, h], None, Lq, n, rope, rotate_k=False)
        O[b, h], lse[b, h] = attention_head(Qh, to_f64(kcache[b, hk, :n]), to_f64(vcache[b, hk, :n]), scale,
                                            causal=True)
    return O, lse
