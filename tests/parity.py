"""Comparison helpers shared by the GPU parity tests.

Tolerances: fp32 scores within 1e-3 relative or 1e-3*max|score| absolute;
indices exact modulo the order of exactly tied scores; V4.1 bf16 scores
within 1 bf16 ulp on >= 99.9% of entries.
"""

import numpy as np
import torch


def score_tol(ref_finite: np.ndarray) -> float:
    m = float(np.abs(ref_finite).max()) if ref_finite.size else 0.0
    return 1e-3 * max(m, 1e-30)


def assert_scores_close(got, ref, what="scores"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: finite pattern differs"
    assert (got[~fin] == ref[~fin]).all(), f"{what}: masked entries differ"
    if fin.any():
        atol = score_tol(ref[fin])
        err = np.abs(got[fin] - ref[fin])
        ok = (err <= atol) | (err <= 1e-3 * np.abs(ref[fin]))
        assert ok.all(), f"{what}: max err {err.max():.3e} > tol {atol:.3e}"


def check_selection_vs_oracle(gidx, gsc, olg, ks, ke, topk, rows_s):
    """GPU selection (indices+scores of each row) against oracle logits.

    gidx/gsc: [n, topk]; olg: oracle logits [n, Skv] (fp64); rows_s: query
    position s of each row.  The selected sets may differ only among keys whose
    oracle scores lie within tolerance of the row's k-th oracle score.
    """
    fin = np.isfinite(olg)
    tol = score_tol(olg[fin]) if fin.any() else 0.0
    for i, s in enumerate(rows_s):
        lo, hi = max(int(ks[s]), 0), min(int(ke[s]), olg.shape[1])
        n = max(hi - lo, 0)
        m = min(n, topk)
        gi = gidx[i]
        assert (gi[m:] == -1).all(), f"row {s}: padding indices"
        assert np.isneginf(gsc[i, m:]).all(), f"row {s}: padding scores"
        sel = gi[:m]
        assert len(set(sel.tolist())) == m, f"row {s}: duplicate indices"
        assert ((sel >= lo) & (sel < hi)).all(), f"row {s}: index out of range"
        assert (np.diff(gsc[i, :m]) <= 0).all(), f"row {s}: not sorted"
        if m == 0:
            continue
        ov = olg[i, sel]
        err = np.abs(gsc[i, :m] - ov)
        assert ((err <= tol) | (err <= 1e-3 * np.abs(ov))).all(), f"row {s}: scores off oracle"
        row = olg[i, lo:hi]
        kth = np.sort(row)[::-1][m - 1]
        # every selected key is within tol of the cut; every unselected one is not clearly above it
        assert (ov >= kth - 2 * tol).all(), f"row {s}: selected a key clearly below the k-th"
        mask = np.ones(n, bool)
        mask[sel - lo] = False
        if mask.any():
            assert (row[mask] <= kth + 2 * tol).all(), f"row {s}: missed a key clearly above the k-th"


def exact_selection_on(logits_rows, ks, ke, topk, rows_s, oracle_mod):
    """Oracle top-k run on the kernel's own fp32 logits (bit-exact reference)."""
    lg = np.asarray(logits_rows, np.float64)
    S = int(max(rows_s)) + 1
    idx, sc = oracle_mod.topk_rows(lg, S, ks, ke, topk, np.asarray(rows_s, np.int64))
    return idx, sc


def bf16_ulp_diff(a_f32: np.ndarray, b_f32: np.ndarray) -> np.ndarray:
    """Distance in bf16 units in the last place between bf16 values held as float32."""
    def key(x):
        u = np.asarray(x, np.float32).view(np.uint32) >> 16
        u = u.astype(np.int64)
        return np.where(u & 0x8000, -(u & 0x7FFF), u)
    return np.abs(key(a_f32) - key(b_f32))
