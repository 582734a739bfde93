"""Tolerances shared by the GPU parity tests.

O: max-abs error <= 2e-2 and relative L2 error <= 1e-2 against the fp64
oracle; lse: |error| <= 1e-3 * max(1, |lse|) (a pure relative bound is
ill-conditioned where lse is near 0, e.g. the first causal row).  Rows the
oracle marks with lse = -inf (no visible key) must come back as -inf with O = 0.
"""
import numpy as np

O_MAX_ABS = 2e-2
O_REL_L2 = 1e-2
LSE_TOL = 1e-3


def to_np(t):
    if hasattr(t, "detach"):
        t = t.detach().float().cpu().numpy()
    return np.asarray(t, dtype=np.float64)


def assert_attn_close(O, lse, O_ref, lse_ref, what=""):
    O, O_ref = to_np(O), np.asarray(O_ref, dtype=np.float64)
    assert O.shape == O_ref.shape, (O.shape, O_ref.shape)
    assert np.isfinite(O).all(), f"{what}: non-finite O"
    err = np.abs(O - O_ref)
    max_abs = float(err.max()) if err.size else 0.0
    denom = float(np.linalg.norm(O_ref))
    rel = float(np.linalg.norm(O - O_ref) / denom) if denom > 0 else float(np.linalg.norm(O - O_ref))
    assert max_abs <= O_MAX_ABS, f"{what}: O max-abs {max_abs:.3e} > {O_MAX_ABS}"
    assert rel <= O_REL_L2, f"{what}: O rel-L2 {rel:.3e} > {O_REL_L2}"
    if lse is not None:
        lse, lse_ref = to_np(lse), np.asarray(lse_ref, dtype=np.float64)
        assert lse.shape == lse_ref.shape
        empty = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(lse), empty), f"{what}: -inf pattern of lse differs"
        d = np.abs(lse[~empty] - lse_ref[~empty])
        bound = LSE_TOL * np.maximum(1.0, np.abs(lse_ref[~empty]))
        worst = float((d / bound).max()) if d.size else 0.0
        assert worst <= 1.0, f"{what}: lse error {worst:.2f}x the bound"
    return max_abs, rel
