"""Literal pure-Python loop form of attention, for tiny shapes only.

TEST INFRASTRUCTURE ONLY (see ``oracle/sdpa.py``).  It is a second,
independent writing of the same definition -- Operator Fusion (GPU learning
diary day 24) §3.4, standard chain ``S = QK^T/sqrt(d) + mask; P = softmax(S);
O = PV`` -- with every sum and exponential spelled out element by element in
Python floats and ``math.exp`` / ``math.log``.  It uses no numpy arithmetic, so
a mistake in the vectorised oracle (a transposed operand, a wrong axis, a
broadcast slip) shows up as a disagreement between the two.
"""
from __future__ import annotations

import math


def _as_nested(x):
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().tolist()
    elif hasattr(x, "tolist"):
        x = x.tolist()
    return x


def attention_loops(q, k, v, scale, causal):
    """q [B][Hq][Lq][D], k/v [B][Hkv][Lkv][D] as nested lists (or arrays).

    Returns (O, lse) as nested lists with the same conventions as the
    vectorised oracle (bottom-right causal alignment, contiguous GQA groups,
    O = 0 and lse = -inf for a row that sees no key).
    """
    q, k, v = _as_nested(q), _as_nested(k), _as_nested(v)
    B, Hq, Lq, D = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    Hkv, Lkv, Dv = len(k[0]), len(k[0][0]), len(v[0][0][0])
    group = Hq // Hkv
    O = [[[[0.0] * Dv for _ in range(Lq)] for _ in range(Hq)] for _ in range(B)]
    lse = [[[0.0] * Lq for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        for h in range(Hq):
            hk = h // group
            for i in range(Lq):
                logits = []
                for j in range(Lkv):
                    if causal and j > i + (Lkv - Lq):
                        continue
                    dot = 0.0
                    for d in range(D):
                        dot += q[b][h][i][d] * k[b][hk][j][d]
                    logits.append((j, scale * dot))
                if not logits:
                    lse[b][h][i] = -math.inf
                    continue
                mx = max(s for _, s in logits)
                denom = 0.0
                for _, s in logits:
                    denom += math.exp(s - mx)
                for j, s in logits:
                    w = math.exp(s - mx) / denom
                    for d in range(Dv):
                        O[b][h][i][d] += w * v[b][hk][j][d]
                lse[b][h][i] = mx + math.log(denom)
    return O, lse
