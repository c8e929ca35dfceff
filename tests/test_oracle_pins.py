"""Pins for the CPU oracle: checks against facts fixed by the indexer pages and
by mathematics, chosen so that a dropped term, a wrong sign or index, or a
transposed operand anywhere in the oracle fails at least one of them.

None of these tests re-derives the oracle's own loops: they use hand-worked
golden values, closed forms, library routines (numpy matmul / sort, torch's
bf16 conversion) on special cases, invariants, and exact finite differences.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def f32(t):
    return t.float().numpy().astype(np.float64)


def bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)


# ----------------------------------------------------------------- causal ranges
def test_causal_ranges_golden():
    for line in open(os.path.join(GOLD, "causal_ranges.txt")):
        if line.startswith("#") or not line.strip():
            continue
        lhs, rhs = line.split(":")
        S, Skv, r = map(int, lhs.split())
        want = [int(x) for x in rhs.split()]
        ks, ke = oracle.causal_ranges(S, Skv, r)
        assert list(ke) == want, (S, Skv, r)
        assert (ks == 0).all()


@pytest.mark.parametrize("name,total", [("tiny", 8128), ("c4_fwd", 2096128),
                                         ("long_fused", 33550336), ("bwd", 8386560)])
def test_causal_visible_pair_counts(name, total):
    # closed form: sum_s min((s+1)//r, Skv) = visible pairs per batch element
    wl = workloads.WORKLOADS[name]
    ks, ke = oracle.causal_ranges(wl.S, wl.Skv, wl.ratio)
    assert int((ke - ks).sum()) == total
    s = np.arange(wl.S)
    assert int(np.minimum((s + 1) // wl.ratio, wl.Skv).sum()) == total


def test_logits_mask_is_prefix():
    wl = workloads.WORKLOADS["tiny"]
    q, k, w = workloads.v4_inputs(wl, 0)
    ks, ke = oracle.causal_ranges(wl.S, wl.Skv, wl.ratio)
    lg = oracle.logits_rows(q, k, w, ks, ke)
    fin = np.isfinite(lg)
    assert fin.sum() == 8128
    for s in range(wl.S):
        assert fin[s, :ke[s]].all() and not fin[s, ke[s]:].any()
    assert (lg[~fin] == -np.inf).all()
    assert not fin[:3].any()  # rows 0..2 see no complete group


def test_logits_general_ranges():
    # explicit [ks, ke) per row (the per-sample interface's cu_seqlen_ks/ke)
    q, k, w = workloads.v4_inputs(workloads.WORKLOADS["tiny"].with_(S=16, Skv=20), 3)
    ks = np.array([0, 2, 5, 7, 0, 19, 3, 3, 10, 0, 1, 2, 3, 4, 5, 6], np.int32)
    ke = np.array([20, 9, 5, 6, 1, 20, 25, 4, 11, 0, 2, 20, 13, 4, 15, 16], np.int32)
    lg = oracle.logits_rows(q, k, w, ks, ke)
    for s in range(16):
        lo, hi = max(ks[s], 0), min(ke[s], 20)
        fin = np.isfinite(lg[s])
        assert fin[lo:hi].all() and fin.sum() == max(hi - lo, 0)


# ------------------------------------------------------------------ scoring
def _full(ke_val, S):
    return np.zeros(S, np.int32), np.full(S, ke_val, np.int32)


def test_identity_single_head_is_matmul():
    # act = identity, H = 1, w = 1  =>  logits = q k^T (numpy matmul)
    g = np.random.default_rng(5)
    S, Skv, D = 24, 40, 32
    q = bf16(g.standard_normal((S, 1, 1, D)))
    k = bf16(g.standard_normal((Skv, 1, D)))
    w = torch.ones(S, 1, 1)
    ks, ke = _full(Skv, S)
    lg = oracle.logits_rows(q, k, w, ks, ke, act="identity")
    ref = f32(q).reshape(S, D) @ f32(k).reshape(Skv, D).T
    np.testing.assert_allclose(lg, ref, rtol=1e-12, atol=1e-12)


def test_relu_on_positive_inputs_is_weighted_matmul():
    # all q, k > 0 => ReLU is the identity => score = (sum_h w_h q_h) . k
    g = np.random.default_rng(6)
    S, Skv, H, D, B = 10, 12, 4, 16, 2
    q = bf16(np.abs(g.standard_normal((S, B, H, D))) + 0.01)
    k = bf16(np.abs(g.standard_normal((Skv, B, D))) + 0.01)
    w = torch.from_numpy(g.standard_normal((S, B, H)).astype(np.float32))
    ks, ke = _full(Skv, S)
    lg = oracle.logits_rows(q, k, w, ks, ke)  # rows r = b*S + s
    qw = np.einsum("sbhd,sbh->bsd", f32(q), w.numpy().astype(np.float64))
    ref = np.einsum("bsd,tbd->bst", qw, f32(k)).reshape(B * S, Skv)
    np.testing.assert_allclose(lg, ref, rtol=1e-11, atol=1e-11)


def test_relu_odd_even_parts():
    # relu(x) - relu(-x) = x ;  relu(x) + relu(-x) = |x|, per head, weighted
    g = np.random.default_rng(7)
    S, Skv, H, D, B = 9, 11, 8, 32, 2
    qf = g.standard_normal((S, B, H, D)).astype(np.float32)
    kf = g.standard_normal((Skv, B, D)).astype(np.float32)
    q, kp, kn = bf16(qf), bf16(kf), bf16(-kf)
    w = torch.from_numpy(g.standard_normal((S, B, H)).astype(np.float32))
    ks, ke = _full(Skv, S)
    lp = oracle.logits_rows(q, kp, w, ks, ke)
    ln = oracle.logits_rows(q, kn, w, ks, ke)
    x = np.einsum("sbhd,tbd->bsht", f32(q), f32(kp))  # numpy contraction
    wb = w.numpy().astype(np.float64).transpose(1, 0, 2)[..., None]  # [B,S,H,1]
    np.testing.assert_allclose(lp - ln, (wb * x).sum(2).reshape(B * S, Skv), rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(lp + ln, (wb * np.abs(x)).sum(2).reshape(B * S, Skv),
                               rtol=1e-10, atol=1e-10)


def test_integer_inputs_are_exact():
    S, Skv, H, D, B = 32, 8, 4, 16, 2
    q, k, w = workloads.integer_inputs(B, S, Skv, H, D, seed=1)
    ks, ke = oracle.causal_ranges(S, Skv, 4)
    lg = oracle.logits_rows(q, k, w, ks, ke)
    x = np.einsum("sbhd,tbd->bsht", f32(q), f32(k))
    ref = (w.numpy().transpose(1, 0, 2)[..., None] * np.maximum(x, 0)).sum(2).reshape(B * S, Skv)
    fin = np.isfinite(lg)
    assert (lg[fin] == ref[fin]).all()
    assert (lg[fin] * 4 == np.round(lg[fin] * 4)).all()  # multiples of 1/4


# -------------------------------------------------------------------- top-k
def _lexsort_topk(row, lo, hi, k):
    t = np.arange(lo, hi)
    v = row[lo:hi]
    order = np.lexsort((t, -v))  # primary: -score, secondary: index
    sel = t[order][:k]
    out = np.full(k, -1, np.int64)
    out[:sel.size] = sel
    return out


@pytest.mark.parametrize("seed", [0, 1])
def test_topk_matches_library_sort(seed):
    wl = workloads.WORKLOADS["tiny"]
    q, k, w = workloads.v4_inputs(wl, seed)
    idx, sc, lg = oracle.indexer_fwd_rows(q, k, w, wl.ratio, wl.topk)
    ks, ke = oracle.causal_ranges(wl.S, wl.Skv, wl.ratio)
    for s in range(wl.S):
        assert (idx[s] == _lexsort_topk(lg[s], ks[s], ke[s], wl.topk)).all()


def test_topk_invariants_and_ties():
    # integer inputs produce many exactly equal scores -> the tie rule matters
    S, Skv, H, D = 64, 16, 4, 16
    q, k, w = workloads.integer_inputs(1, S, Skv, H, D, seed=2)
    k = bf16(np.abs(f32(k)) * 0)  # all keys zero: every visible score is 0.0
    q2, k2, w2 = workloads.integer_inputs(1, S, Skv, H, D, seed=3)
    for qq, kk, ww in ((q, k, w), (q2, k2, w2)):
        topk = 6
        idx, sc, lg = oracle.indexer_fwd_rows(qq, kk, ww, 4, topk)
        ks, ke = oracle.causal_ranges(S, Skv, 4)
        for s in range(S):
            n = ke[s] - ks[s]
            m = min(n, topk)
            sel = idx[s, :m]
            assert (idx[s, m:] == -1).all() and np.isneginf(sc[s, m:]).all()
            assert len(set(sel.tolist())) == m
            assert ((sel >= ks[s]) & (sel < ke[s])).all()
            assert (np.diff(sc[s, :m]) <= 0).all()  # sorted descending
            for a in range(m - 1):  # equal scores in ascending index order
                if sc[s, a] == sc[s, a + 1]:
                    assert sel[a] < sel[a + 1]
            if m:
                rest = np.setdiff1d(np.arange(ks[s], ke[s]), sel)
                assert (lg[s, rest] <= sc[s, m - 1]).all()
                # ties at the boundary: every unselected equal score has a larger index
                eq = rest[lg[s, rest] == sc[s, m - 1]]
                assert (eq > sel[sc[s, :m] == sc[s, m - 1]].max()).all()
            assert (sc[s, :m] == lg[s, sel]).all()
    # all-zero keys: the selection is the first min(topk, n) indices in order
    idx, sc, _ = oracle.indexer_fwd_rows(q, k, w, 4, 6)
    assert (idx[-1] == np.arange(6)).all() and (sc[-1] == 0).all()


def test_topk_larger_than_visible_returns_all():
    wl = workloads.WORKLOADS["tiny"]
    q, k, w = workloads.v4_inputs(wl, 0)
    idx, sc, lg = oracle.indexer_fwd_rows(q, k, w, wl.ratio, 80)
    ks, ke = oracle.causal_ranges(wl.S, wl.Skv, wl.ratio)
    for s in range(wl.S):
        n = ke[s]
        assert sorted(idx[s, :n].tolist()) == list(range(n))
        assert (idx[s, n:] == -1).all()


def test_extract_is_gather():
    wl = workloads.WORKLOADS["tiny"]
    q, k, w = workloads.v4_inputs(wl, 0)
    idx, sc, lg = oracle.indexer_fwd_rows(q, k, w, wl.ratio, wl.topk)
    ex = oracle.extract_rows(lg, idx)
    assert (ex == sc).all()  # bit-exact: same values
    g = np.random.default_rng(0)
    ridx = g.integers(-3, wl.Skv + 3, size=(wl.S, 5)).astype(np.int32)
    ex = oracle.extract_rows(lg, ridx)
    ks, ke = oracle.causal_ranges(wl.S, wl.Skv, wl.ratio)
    for s in range(wl.S):
        for j in range(5):
            t = ridx[s, j]
            want = lg[s, t] if 0 <= t < wl.Skv else -np.inf
            assert ex[s, j] == want
    # the sparse gather agrees with the dense logits at the same indices
    gs = oracle.gather_scores_rows(q, k, w, ks, ke, ridx)
    assert np.array_equal(gs, ex)


# --------------------------------------------------------------------- bf16
def test_bf16_round_golden():
    for line in open(os.path.join(GOLD, "bf16_rounding.txt")):
        if line.startswith("#") or not line.strip():
            continue
        a, b = line.split()
        assert oracle.bf16_round([float.fromhex(a)])[0] == float.fromhex(b), a


def test_bf16_round_matches_torch_conversion():
    g = np.random.default_rng(9)
    bits = g.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    ours = oracle.bf16_round(v.astype(np.float64))
    ref = torch.from_numpy(v.copy()).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(ours, ref)


# --------------------------------------------------------------------- V4.1
def test_v41_exact_case_reduces_to_plain_score():
    # integer inputs with D=16 keep q.k integral and |q.k| <= 64, and w in
    # {+-1/4,+-1/2,+-1}: both intermediate roundings are exact, so the result
    # is bf16(exact weighted ReLU sum).  The final rounding is the library's.
    B, S, Skv, H, D = 2, 12, 10, 4, 16
    q, k, w = workloads.integer_inputs(B, S, Skv, H, D, seed=4, layout="bshd")
    wb = w.to(torch.bfloat16)
    allowed = torch.from_numpy(np.random.default_rng(1).random((B, S, Skv)) < 0.7)
    out = oracle.scores_v41_rows(q, k, wb, allowed).reshape(B, S, Skv)
    x = np.einsum("bshd,btd->bsht", f32(q), f32(k))
    exact = (np.maximum(x, 0) * f32(wb)[..., None]).sum(2)
    ref = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16).float().numpy()
    al = allowed.numpy()
    assert np.array_equal(out[al], ref[al])
    assert np.isneginf(out[~al]).all()


def test_v41_rounds_gemm_result_and_weighted_score():
    # q,k = j/8 with |j| <= 15, D = 32: q.k is exact in float32 (multiples of
    # 2^-6 below 2^13) but not in bf16, so each rounding step is exercised.
    g = np.random.default_rng(10)
    B, S, Skv, H, D = 1, 6, 7, 2, 32
    q = bf16(g.integers(-15, 16, (B, S, H, D)) / 8.0)
    k = bf16(g.integers(-15, 16, (B, Skv, D)) / 8.0)
    allowed = torch.ones(B, S, Skv, dtype=torch.bool)
    x = np.einsum("bshd,btd->bsht", f32(q), f32(k)).astype(np.float32)  # exact
    y = torch.from_numpy(x).to(torch.bfloat16).float()                   # library RNE
    for wv in (1.0, 0.75, -0.375):
        w = torch.full((B, S, H), wv).to(torch.bfloat16)
        zz = (torch.relu(y) * wv).to(torch.bfloat16).double()            # exact product, RNE
        ref = zz.sum(2).float().to(torch.bfloat16).float().numpy()
        out = oracle.scores_v41_rows(q, k, w, allowed, act="relu").reshape(B, S, Skv)
        assert np.array_equal(out, ref), wv
        xi = torch.from_numpy(x)
        yi = xi.to(torch.bfloat16).float()
        zi = (yi * wv).to(torch.bfloat16).double().sum(2).float().to(torch.bfloat16).float()
        out_id = oracle.scores_v41_rows(q, k, w, allowed, act="identity").reshape(B, S, Skv)
        assert np.array_equal(out_id, zi.numpy()), wv


def test_v41_all_false_row_is_neg_inf():
    B, S, Skv, H, D = 1, 4, 9, 2, 16
    q, k, w = workloads.integer_inputs(B, S, Skv, H, D, seed=5, layout="bshd")
    allowed = torch.zeros(B, S, Skv, dtype=torch.bool)
    out = oracle.scores_v41_rows(q, k, w.to(torch.bfloat16), allowed)
    assert np.isneginf(out).all()


# ----------------------------------------------------------------- backward
def _bwd_case(seed=0, S=48, Skv=12, H=4, D=16, topk=5, B=2, grid=True):
    g = np.random.default_rng(seed)
    # values on a 1/16 grid so that +-1/16 steps are exact in bf16
    q = bf16(g.integers(-24, 25, (S, B, H, D)) / 16.0) if grid else bf16(g.standard_normal((S, B, H, D)))
    k = bf16(g.integers(-24, 25, (Skv, B, D)) / 16.0) if grid else bf16(g.standard_normal((Skv, B, D)))
    w = torch.from_numpy(g.standard_normal((S, B, H)).astype(np.float32))
    ks, ke = oracle.causal_ranges(S, Skv, 4)
    n = ke - ks
    idx = workloads.random_selection(B, S, Skv, topk, n, seed).numpy()
    # the layout of idx/grad is [B,S,topk]; rows r = b*S + s
    grad = workloads.grad_scores(B, S, topk, seed).numpy()
    return q, k, w, idx, grad, ks, ke


def _loss(q, k, w, idx, grad, ks, ke, act="relu"):
    S, B = q.shape[0], q.shape[1]
    sc = oracle.gather_scores_rows(q, k, w, ks, ke, idx.reshape(B * S, -1), act=act)
    valid = np.isfinite(sc)
    return float((np.where(valid, sc, 0.0) * grad.reshape(B * S, -1)).sum())


def test_bwd_exact_central_differences():
    """The loss L = sum g*score is piecewise linear in each q and k entry; a
    +-1/16 step that crosses no ReLU kink gives the derivative exactly."""
    q, k, w, idx, grad, ks, ke = _bwd_case()
    dq, dk, dw, *_ = oracle.bwd(q, k, w, idx, grad, ks, ke)
    S, B, H, D = q.shape
    qf, kf = f32(q), f32(k)
    x = np.einsum("sbhd,tbd->sbht", qf, kf)
    g = np.random.default_rng(1)
    step = 1.0 / 16
    checked = 0
    for _ in range(120):
        s, b, h, d = (int(g.integers(0, n)) for n in (S, B, H, D))
        if np.abs(x[s, b, h, :]).min() <= step * np.abs(kf[:, b, d]).max():
            continue  # a kink could be crossed
        qp, qm = qf.copy(), qf.copy()
        qp[s, b, h, d] += step
        qm[s, b, h, d] -= step
        fd = (_loss(bf16(qp), k, w, idx, grad, ks, ke) - _loss(bf16(qm), k, w, idx, grad, ks, ke)) / (2 * step)
        assert abs(fd - dq[s, b, h, d]) <= 1e-9 * (1 + abs(fd)), (s, b, h, d)
        checked += 1
    assert checked > 20
    checked = 0
    for t in range(k.shape[0]):
        for b in range(B):
            d = int(g.integers(0, D))
            if np.abs(x[:, b, :, t]).min() <= step * np.abs(qf[:, b, :, d]).max():
                continue
            kp, km = kf.copy(), kf.copy()
            kp[t, b, d] += step
            km[t, b, d] -= step
            fd = (_loss(q, bf16(kp), w, idx, grad, ks, ke) - _loss(q, bf16(km), w, idx, grad, ks, ke)) / (2 * step)
            assert abs(fd - dk[t, b, d]) <= 1e-9 * (1 + abs(fd)), (t, b, d)
            checked += 1
    # dw: the loss is exactly linear in w
    wf = w.numpy().astype(np.float64)
    for _ in range(40):
        s, b, h = (int(g.integers(0, n)) for n in (S, B, H))
        wp, wm = wf.copy(), wf.copy()
        wp[s, b, h] += 0.25
        wm[s, b, h] -= 0.25
        fd = (_loss(q, k, torch.from_numpy(wp.astype(np.float32)), idx, grad, ks, ke)
              - _loss(q, k, torch.from_numpy(wm.astype(np.float32)), idx, grad, ks, ke)) / 0.5
        assert abs(fd - dw[s, b, h]) <= 1e-6 * (1 + abs(fd))


def test_bwd_euler_homogeneity():
    # score is degree-1 homogeneous in w, in q and in k (ReLU or identity):
    # per row sum_h w*dw = sum_{h,d} q*dq = sum_j g*score; globally sum k*dk = sum g*score
    for act in ("relu", "identity"):
        q, k, w, idx, grad, ks, ke = _bwd_case(seed=3, grid=False)
        S, B, H, D = q.shape
        dq, dk, dw, *_ = oracle.bwd(q, k, w, idx, grad, ks, ke, act=act)
        sc = oracle.gather_scores_rows(q, k, w, ks, ke, idx.reshape(B * S, -1), act=act)
        gs = (np.where(np.isfinite(sc), sc, 0) * grad.reshape(B * S, -1)).sum(1).reshape(B, S)
        wf, qf, kf = w.numpy().astype(np.float64), f32(q), f32(k)
        np.testing.assert_allclose((wf * dw).sum(2).T, gs, rtol=1e-9, atol=1e-9)
        np.testing.assert_allclose((qf * dq).sum((2, 3)).T, gs, rtol=1e-9, atol=1e-9)
        np.testing.assert_allclose((kf * dk).sum(), gs.sum(), rtol=1e-9, atol=1e-9)


def test_bwd_padding_and_invisible_get_no_gradient():
    q, k, w, idx, grad, ks, ke = _bwd_case(seed=4)
    S, B = q.shape[0], q.shape[1]
    idx2 = idx.copy()
    g2 = grad.copy()
    # point every padding slot at a key past the row's range: still no gradient
    for b in range(B):
        for s in range(S):
            pad = idx2[b, s] < 0
            idx2[b, s, pad] = min(int(ke[s]) + 1, k.shape[0] - 1) if ke[s] + 1 < k.shape[0] else -1
            g2[b, s, pad] = 123.0
    a = oracle.bwd(q, k, w, idx, grad, ks, ke)
    c = oracle.bwd(q, k, w, idx2, np.where(idx < 0, g2, grad), ks, ke)
    for x, y in zip(a[:3], c[:3]):
        assert np.array_equal(x, y)


def test_bwd_identity_closed_form():
    # identity activation: dq[s,b,h,:] = w[s,b,h] * sum_j g_j k[idx_j, b, :]
    q, k, w, idx, grad, ks, ke = _bwd_case(seed=5, grid=False)
    S, B, H, D = q.shape
    dq, dk, dw, *_ = oracle.bwd(q, k, w, idx, grad, ks, ke, act="identity")
    kf = f32(k)
    for b in range(B):
        for s in range(S):
            sel = idx[b, s] >= 0
            gk = (grad[b, s, sel][:, None] * kf[idx[b, s, sel], b, :]).sum(0)
            np.testing.assert_allclose(dq[s, b], w.numpy()[s, b][:, None] * gk, rtol=1e-10, atol=1e-12)


# ------------------------------------------------------------ masked top-k
def test_topk_masked_matches_library_sort():
    """Selection over arbitrary visible sets: numpy lexsort over the visible
    entries of each row (ties included), padding past the visible count."""
    g = np.random.default_rng(12)
    n, Skv, topk = 40, 70, 24
    lg = g.integers(-4, 5, (n, Skv)).astype(np.float64) * 0.5  # many exact ties
    mask = (g.random((n, Skv)) < np.linspace(0.05, 0.9, n)[:, None]).astype(np.uint8)
    idx, sc = oracle.topk_masked_rows(lg, mask, topk)
    for i in range(n):
        t = np.flatnonzero(mask[i])
        order = np.lexsort((t, -lg[i, t]))
        sel = t[order][:topk]
        assert (idx[i, :sel.size] == sel).all() and (idx[i, sel.size:] == -1).all()
        assert (sc[i, :sel.size] == lg[i, sel]).all() and np.isneginf(sc[i, sel.size:]).all()


def test_topk_masked_contiguous_mask_equals_range_topk():
    wl = workloads.WORKLOADS["tiny"]
    q, k, w = workloads.v4_inputs(wl, 1)
    ks, ke = oracle.causal_ranges(wl.S, wl.Skv, wl.ratio)
    idx, sc, lg = oracle.indexer_fwd_rows(q, k, w, wl.ratio, wl.topk)
    mask = (np.arange(wl.Skv)[None, :] < ke[:, None]).astype(np.uint8)
    midx, msc = oracle.topk_masked_rows(np.nan_to_num(lg, neginf=0.0), mask, wl.topk)
    assert np.array_equal(midx, idx) and np.array_equal(msc, sc)


# ------------------------------------------------------ backward slack outputs
def _slack_case(act):
    """One row (s = 7, ratio 1) selecting key 0 with q.k = 0 exactly and key 1
    with q.k = 3; H = 1, D = 16, w = 0.75, grads 0.5 and 2."""
    S, Skv, D = 8, 2, 16
    q = np.zeros((S, 1, 1, D), np.float32)
    k = np.zeros((Skv, 1, D), np.float32)
    q[7, 0, 0, :2] = [1, 1]
    k[0, 0, :2] = [1, -1]
    k[1, 0, :2] = [2, 1]
    w = torch.full((S, 1, 1), 0.75)
    idx = np.full((1, S, 2), -1, np.int32)
    idx[0, 7] = [0, 1]
    grad = np.zeros((1, S, 2), np.float32)
    grad[0, 7] = [0.5, 2.0]
    ks, ke = oracle.causal_ranges(S, Skv, 1)
    return oracle.bwd(bf16(q), bf16(k), w, idx, grad, ks, ke, act=act), D


def test_bwd_slack_marks_exactly_the_ambiguous_relu_pair():
    (dq, dk, dw, sq, sk, sw), D = _slack_case("relu")
    gamma = D * 2.0 ** -22
    # ReLU'(0) = 0: only key 1 reaches dq and dk; dw = 0.5*relu(0) + 2*3
    assert np.array_equal(dq[7, 0, 0, :3], [3.0, 1.5, 0.0]) and dw[7, 0, 0] == 6.0
    assert np.array_equal(dk[0, 0, :3], [0, 0, 0]) and np.array_equal(dk[1, 0, :3], [1.5, 1.5, 0])
    # the x = 0 pair widens the bound by |g w| |k| on dq, |g w| |q| on dk, |g| gamma sum|q k| on dw
    assert np.array_equal(sq[7, 0, 0, :3], [0.375, 0.375, 0.0])
    assert np.array_equal(sk[0, 0, :3], [0.375, 0.375, 0.0]) and (sk[1] == 0).all()
    assert sw[7, 0, 0] == 0.5 * gamma * 2.0
    sq[7, 0, 0, :2] = 0
    sk[0, 0, :2] = 0
    sw[7, 0, 0] = 0
    assert not sq.any() and not sk.any() and not sw.any()


def test_bwd_slack_is_zero_for_identity_and_far_from_kinks():
    (dq, dk, dw, sq, sk, sw), _ = _slack_case("identity")
    assert not sq.any() and not sk.any() and not sw.any()
    assert np.array_equal(dq[7, 0, 0, :3], [0.75 * (0.5 * 1 + 2 * 2), 0.75 * (0.5 * -1 + 2 * 1), 0])
    # all-positive queries and keys: every |x| is far above gamma * sum|q k|
    q, k, w, idx, grad, ks, ke = _bwd_case(seed=6)
    q, k = bf16(np.abs(f32(q)) + 0.5), bf16(np.abs(f32(k)) + 0.5)
    *_, sq, sk, sw = oracle.bwd(q, k, w, idx, grad, ks, ke)
    assert not sq.any() and not sk.any() and not sw.any()
