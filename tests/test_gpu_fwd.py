"""GPU parity of the V4 forward (scoring, causal mask, top-k) against the CPU
oracle, through the C ABI."""

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_top_tcgen05_gb300 as lidx
import workloads
from parity import (assert_scores_close, check_selection_vs_oracle, exact_selection_on,
                    score_tol)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_attention_top_tcgen05_gb300 import build

    build.build()
    lidx.lib()
    yield
    assert lidx.lidx_device_status() == 0


def cuda(*ts):
    return [t.to(DEV) for t in ts]


def run_fwd(q, k, w, ratio, topk, materialise, act="relu"):
    qd, kd, wd = cuda(q, k, w)
    idx, sc, lg = lidx.lidx_indexer_fwd(qd, kd, wd, ratio, topk, act=act,
                                        materialise_logits=materialise)
    torch.cuda.synchronize()
    assert lidx.lidx_device_status() == 0
    return idx.cpu().numpy(), sc.cpu().numpy(), None if lg is None else lg.cpu().numpy()


def full_check(q, k, w, ratio, topk, act="relu", materialise=True, rows=None):
    S, B, H, D = q.shape
    Skv = k.shape[0]
    idx, sc, lg = run_fwd(q, k, w, ratio, topk, materialise, act)
    ks, ke = oracle.causal_ranges(S, Skv, ratio)
    r = np.arange(B * S) if rows is None else np.asarray(rows)
    olg = oracle.logits_rows(q, k, w, ks, ke, act, r)
    rs = r % S
    gidx = idx.reshape(B * S, topk)[r]
    gsc = sc.reshape(B * S, topk)[r]
    if lg is not None:
        glg = lg.reshape(B * S, Skv)[r]
        assert_scores_close(glg, olg, "logits")
        eidx, esc = exact_selection_on(glg, ks, ke, topk, rs, oracle)
        assert np.array_equal(gidx, eidx), "selection differs from exact top-k of the kernel's logits"
        assert np.array_equal(gsc.astype(np.float64), esc)
    check_selection_vs_oracle(gidx, gsc, olg, ks, ke, topk, rs)
    return idx, sc, lg


def test_identity_single_head_matches_library_gemm():
    # act = identity, H = 1, w = 1, full ranges: logits are q k^T
    g = np.random.default_rng(0)
    S, Skv, D = 600, 300, 64
    q = workloads.to_bf16(g.standard_normal((S, 1, 1, D)).astype(np.float32))
    k = workloads.to_bf16(g.standard_normal((Skv, 1, D)).astype(np.float32))
    w = torch.ones(S, 1, 1)
    qd, kd, wd = cuda(q, k, w)
    ks = torch.zeros(S, dtype=torch.int32, device=DEV)
    ke = torch.full((S,), Skv, dtype=torch.int32, device=DEV)
    lg = lidx.lidx_indexer_logits(qd, kd, wd, 1, ks, ke, clean=True, act="identity")
    ref = (qd.float().reshape(S, D) @ kd.float().reshape(Skv, D).T)
    torch.cuda.synchronize()
    err = (lg.reshape(S, Skv) - ref).abs().max().item()
    assert err <= 1e-3 * ref.abs().max().item(), err
    olg = oracle.logits_rows(q, k, w, np.zeros(S, np.int32), np.full(S, Skv, np.int32), "identity")
    assert_scores_close(lg.cpu().numpy().reshape(S, Skv), olg)


@pytest.mark.parametrize("H,D", [(8, 32), (64, 128), (128, 64), (4, 16), (16, 48)])
def test_integer_inputs_bit_exact(H, D):
    # every partial sum is exact in fp32, so the kernel must equal the oracle bit for bit
    B, S, Skv = 2, 200, 150
    q, k, w = workloads.integer_inputs(B, S, Skv, H, D, seed=H + D)
    qd, kd, wd = cuda(q, k, w)
    lg = lidx.lidx_indexer_logits(qd, kd, wd, 1).cpu().numpy().reshape(B * S, Skv)
    ks, ke = oracle.causal_ranges(S, Skv, 1)
    olg = oracle.logits_rows(q, k, w, ks, ke)
    assert np.array_equal(lg, olg.astype(np.float32))


def test_tiny_workload():
    wl = workloads.WORKLOADS["tiny"]
    q, k, w = workloads.v4_inputs(wl, 0)
    idx, sc, lg = full_check(q, k, w, wl.ratio, wl.topk)
    assert np.isfinite(lg).sum() == 8128
    # extract_topk_scores on the kernel's logits returns the selected scores bit-exactly
    ex = lidx.lidx_extract_topk_scores(torch.from_numpy(lg).to(DEV), torch.from_numpy(idx).to(DEV))
    assert np.array_equal(ex.cpu().numpy(), sc)


def test_tiny_identity_act():
    wl = workloads.WORKLOADS["tiny"]
    q, k, w = workloads.v4_inputs(wl, 1)
    full_check(q, k, w, wl.ratio, wl.topk, act="identity")


def test_c4_layer_workload_full():
    wl = workloads.WORKLOADS["c4_fwd"]
    q, k, w = workloads.v4_inputs(wl, 0)
    idx, sc, lg = full_check(q, k, w, wl.ratio, wl.topk)
    assert np.isfinite(lg).sum() == 2096128


@pytest.mark.parametrize("H,D,B,S,Skv,ratio,topk", [
    (64, 128, 2, 1000, 333, 3, 100),    # ragged query tiles and key tiles
    (8, 32, 1, 777, 190, 4, 64),
    (128, 128, 1, 300, 520, 1, 256),     # ratio 1: every earlier key visible, clamp at Skv
    (32, 64, 3, 129, 40, 2, 50),         # topk > visible keys on every row
    (1, 16, 1, 513, 256, 2, 17),
    (2, 48, 2, 260, 70, 4, 5),
    (128, 64, 2, 1000, 300, 2, 40),     # two rows per query tile, several tiles per CTA:
                                         # some selection groups own no row of a tile
])
def test_shapes_fused_and_materialised(H, D, B, S, Skv, ratio, topk):
    g = np.random.default_rng(H * 7 + D)
    q = workloads.to_bf16(g.standard_normal((S, B, H, D)).astype(np.float32) / np.sqrt(D))
    k = workloads.to_bf16(g.standard_normal((Skv, B, D)).astype(np.float32) / np.sqrt(D))
    w = torch.from_numpy((g.standard_normal((S, B, H)) / np.sqrt(H)).astype(np.float32))
    i1, s1, _ = full_check(q, k, w, ratio, topk, materialise=True)
    i2, s2, _ = full_check(q, k, w, ratio, topk, materialise=False)
    # the fused path computes the same fp32 scores: identical results
    assert np.array_equal(i1, i2) and np.array_equal(s1, s2)


def test_explicit_ranges_clean_and_unclean():
    g = np.random.default_rng(3)
    S, B, H, D, Skv = 300, 2, 16, 64, 500
    q = workloads.to_bf16(g.standard_normal((S, B, H, D)).astype(np.float32) / 8)
    k = workloads.to_bf16(g.standard_normal((Skv, B, D)).astype(np.float32) / 8)
    w = torch.from_numpy(g.standard_normal((S, B, H)).astype(np.float32) / 4)
    ks = g.integers(-5, Skv, S).astype(np.int32)
    ke = (ks + g.integers(-3, 300, S)).astype(np.int32)
    qd, kd, wd = cuda(q, k, w)
    ksd, ked = torch.from_numpy(ks).to(DEV), torch.from_numpy(ke).to(DEV)
    lg = lidx.lidx_indexer_logits(qd, kd, wd, 1, ksd, ked, clean=True).cpu().numpy()
    olg = oracle.logits_rows(q, k, w, ks, ke)
    assert_scores_close(lg.reshape(B * S, Skv), olg)
    # clean=False: visible entries are still exact; the rest is unspecified
    sentinel = torch.full((B, S, Skv), 7.0, device=DEV)
    lg2 = lidx.lidx_indexer_logits(qd, kd, wd, 1, ksd, ked, clean=False, out=sentinel)
    lg2 = lg2.cpu().numpy().reshape(B * S, Skv)
    fin = np.isfinite(olg)
    assert np.array_equal(lg2[fin], lg.reshape(B * S, Skv)[fin])


def test_explicit_ranges_short_rows_one_warp_each():
    """Every row spans at most 128 keys (Skv = 120), so each selection warp takes
    rows of its own; explicit ranges, including empty and clamped ones.  The fused
    and materialised calls agree bit for bit, equal the exact top-k of the
    kernel's own logits, and the oracle's within tolerance."""
    g = np.random.default_rng(11)
    S, B, H, D, Skv, topk = 700, 2, 32, 64, 120, 40
    q = workloads.to_bf16(g.standard_normal((S, B, H, D)).astype(np.float32) / np.sqrt(D))
    k = workloads.to_bf16(g.standard_normal((Skv, B, D)).astype(np.float32) / np.sqrt(D))
    w = torch.from_numpy((g.standard_normal((S, B, H)) / np.sqrt(H)).astype(np.float32))
    ks = g.integers(-5, Skv, S).astype(np.int32)
    ke = (ks + g.integers(-3, 90, S)).astype(np.int32)
    qd, kd, wd = cuda(q, k, w)
    ksd, ked = torch.from_numpy(ks).to(DEV), torch.from_numpy(ke).to(DEV)
    i1, s1, lg = lidx.lidx_indexer_fwd_ranges(qd, kd, wd, ksd, ked, topk, materialise_logits=True)
    i2, s2, _ = lidx.lidx_indexer_fwd_ranges(qd, kd, wd, ksd, ked, topk)
    torch.cuda.synchronize()
    assert lidx.lidx_device_status() == 0
    assert torch.equal(i1, i2) and torch.equal(s1, s2)
    glg = lg.cpu().numpy().reshape(B * S, Skv)
    olg = oracle.logits_rows(q, k, w, ks, ke)
    assert_scores_close(glg, olg, "logits")
    rs = np.arange(B * S) % S
    eidx, esc = exact_selection_on(glg, ks, ke, topk, rs, oracle)
    gidx, gsc = i1.cpu().numpy().reshape(B * S, topk), s1.cpu().numpy().reshape(B * S, topk)
    assert np.array_equal(gidx, eidx)
    assert np.array_equal(gsc.astype(np.float64), esc)
    check_selection_vs_oracle(gidx, gsc, olg, ks, ke, topk, rs)


def test_edge_cases():
    g = np.random.default_rng(4)
    # Skv = 0: every row is padding
    q = workloads.to_bf16(g.standard_normal((10, 1, 8, 32)).astype(np.float32))
    k = workloads.to_bf16(np.zeros((0, 1, 32), np.float32))
    w = torch.ones(10, 1, 8)
    idx, sc, _ = run_fwd(q, k, w, 4, 3, False)
    assert (idx == -1).all() and np.isneginf(sc).all()
    # S smaller than one query tile, topk 1
    wl = workloads.WORKLOADS["tiny"].with_(S=5, Skv=3)
    q, k, w = workloads.v4_inputs(wl, 2)
    full_check(q, k, w, 1, 1)
    # all keys zero: every visible score is exactly 0 -> first indices in order
    S, Skv = 64, 16
    q, k, w = workloads.integer_inputs(1, S, Skv, 8, 32, seed=9)
    k = torch.zeros_like(k)
    idx, sc, _ = run_fwd(q, k, w, 4, 6, False)
    assert (idx[0, -1] == np.arange(6)).all() and (sc[0, -1] == 0).all()
    # one outlier key and many exact zeros: one bucket holds almost the whole row
    q, k, w = workloads.integer_inputs(1, 256, 64, 8, 32, seed=11)
    kk = torch.zeros_like(k)
    kk[5] = k[5]
    full_check(q, kk, w, 1, 16)
    # heavy ties from integer inputs: exact comparison on the kernel's logits
    q, k, w = workloads.integer_inputs(2, 400, 100, 8, 32, seed=10)
    full_check(q, k, w, 4, 40)


def test_long_context_fused_sampled_rows():
    """Full-size long-context workload in the benchmark's launch configuration
    (fused, no logits); oracle on a strided sample of rows."""
    wl = workloads.WORKLOADS["long_fused"]
    q, k, w = workloads.v4_inputs(wl, 0)
    rows = workloads.sample_rows(wl.B, wl.S, 509, 3)
    full_check(q, k, w, wl.ratio, wl.topk, materialise=False, rows=rows)


@pytest.mark.parametrize("H,D,B,S,Skv,ratio,topk", [
    (64, 128, 1, 4096, 1024, 4, 512),   # c4-layer shapes, tensor-core path
    (8, 32, 2, 300, 90, 4, 20),         # plain-FMA path
    (128, 64, 1, 200, 6000, 1, 37),     # Skv beyond the selection limit is fine here
])
def test_given_indices_score_only_those_pairs(H, D, B, S, Skv, ratio, topk):
    """topk_indices given: no selection; scores of exactly those pairs, -inf for
    indices outside the row's causal range (padding -1 included)."""
    g = np.random.default_rng(H + S)
    q = workloads.to_bf16(g.standard_normal((S, B, H, D)).astype(np.float32) / np.sqrt(D))
    k = workloads.to_bf16(g.standard_normal((Skv, B, D)).astype(np.float32) / np.sqrt(D))
    w = torch.from_numpy((g.standard_normal((S, B, H)) / np.sqrt(H)).astype(np.float32))
    ks, ke = oracle.causal_ranges(S, Skv, ratio)
    idx = workloads.random_selection(B, S, Skv, topk, ke - ks, 2).numpy()
    junk = g.random(idx.shape) < 0.05  # some indices past the range or negative
    idx[junk] = g.integers(-3, Skv + 3, int(junk.sum()))
    qd, kd, wd = cuda(q, k, w)
    idd = torch.from_numpy(idx).to(DEV)
    ref = oracle.gather_scores_rows(q, k, w, ks, ke, idx.reshape(B * S, topk))
    for materialise in (False, True):
        oi, osc, _ = lidx.lidx_indexer_fwd(qd, kd, wd, ratio, topk, topk_indices=idd,
                                           materialise_logits=materialise)
        torch.cuda.synchronize()
        assert lidx.lidx_device_status() == 0
        assert np.array_equal(oi.cpu().numpy(), idx)
        assert_scores_close(osc.cpu().numpy().reshape(B * S, topk), ref, "given-index scores")


@pytest.mark.parametrize("B,S,Skv,ratio,topk", [(1, 5000, 1250, 4, 512), (2, 2100, 1100, 1, 1024)])
def test_fused_only_configuration(B, S, Skv, ratio, topk):
    """D = 128, ReLU, Skv > 1024 and no logits: the fused call runs the fused-only
    build, the materialised one the general build.  Both compute the same fp32
    scores, so their results are identical, and they equal the oracle."""
    g = np.random.default_rng(S + Skv)
    H, D = 64, 128
    q = workloads.to_bf16(g.standard_normal((S, B, H, D)).astype(np.float32) / np.sqrt(D))
    k = workloads.to_bf16(g.standard_normal((Skv, B, D)).astype(np.float32) / np.sqrt(D))
    w = torch.from_numpy((g.standard_normal((S, B, H)) / np.sqrt(H)).astype(np.float32))
    rows = np.concatenate([np.arange(0, B * S, 37), [S - 1, B * S - 1]])  # the oracle on a sample
    i1, s1, _ = full_check(q, k, w, ratio, topk, materialise=True, rows=rows)
    i2, s2, _ = run_fwd(q, k, w, ratio, topk, False)
    assert np.array_equal(i1, i2) and np.array_equal(s1, s2)


def test_fused_forward_beyond_one_selection_window():
    """Rows with more visible keys than one shared-memory window of candidates
    (Skv 9000, ratio 1): the fused and materialised paths agree, the selection
    equals the exact top-k of the kernel's own logits, and sampled rows agree
    with the oracle."""
    g = np.random.default_rng(21)
    S, B, H, D, Skv, topk = 9100, 1, 8, 32, 9000, 4500
    q = workloads.to_bf16(g.standard_normal((S, B, H, D)).astype(np.float32) / np.sqrt(D))
    k = workloads.to_bf16(g.standard_normal((Skv, B, D)).astype(np.float32) / np.sqrt(D))
    w = torch.from_numpy((g.standard_normal((S, B, H)) / np.sqrt(H)).astype(np.float32))
    rows = np.concatenate([np.arange(0, S, 397), [4499, 4500, 8999, S - 1]])
    i1, s1, _ = full_check(q, k, w, 1, topk, materialise=True, rows=rows)
    i2, s2, _ = run_fwd(q, k, w, 1, topk, False)
    assert np.array_equal(i1, i2) and np.array_equal(s1, s2)


def test_given_indices_without_keys_are_copied():
    g = np.random.default_rng(6)
    S, B, H, D, topk = 20, 2, 8, 32, 5
    q = workloads.to_bf16(g.standard_normal((S, B, H, D)).astype(np.float32))
    k = workloads.to_bf16(np.zeros((0, B, D), np.float32))
    w = torch.ones(S, B, H)
    idx = torch.from_numpy(g.integers(-2, 9, (B, S, topk)).astype(np.int32))
    qd, kd, wd = cuda(q, k, w)
    oi, osc, _ = lidx.lidx_indexer_fwd(qd, kd, wd, 4, topk, topk_indices=idx.to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(oi.cpu().numpy(), idx.numpy()) and np.isneginf(osc.cpu().numpy()).all()


@pytest.mark.parametrize("ranks", [2, 3])
def test_context_parallel_shards_on_the_cuda_path(ranks):
    """Host-simulated context-parallel ranks: each holds a contiguous shard of
    query rows (global positions p0..p0+S_r) and every compressed key, and calls
    the library with its own causal ranges.  The shards' forward outputs
    concatenate to the unsharded call bit for bit; their dq equals the
    unsharded one bit for bit and their dw up to fp32 reassociation, and their
    partial dk sum to the full dk."""
    wl = workloads.WORKLOADS["c4_fwd"].with_(S=2048, Skv=512, topk=256)
    q, k, w = workloads.v4_inputs(wl, 4)
    qd, kd, wd = cuda(q, k, w)
    S, ratio, topk = wl.S, wl.ratio, wl.topk
    full_i, full_s, _ = lidx.lidx_indexer_fwd(qd, kd, wd, ratio, topk)
    grad = workloads.grad_scores(1, S, topk, 4).to(DEV)
    fdq, fdk, fdw = lidx.lidx_indexer_bwd(qd, kd, wd, full_i, grad, ratio)
    cuts = np.linspace(0, S, ranks + 1).astype(int)
    dk_sum = torch.zeros_like(fdk)
    for r in range(ranks):
        p0, p1 = int(cuts[r]), int(cuts[r + 1])
        pos = np.arange(p0, p1)
        ks = torch.zeros(p1 - p0, dtype=torch.int32, device=DEV)
        ke = torch.from_numpy(np.minimum((pos + 1) // ratio, wl.Skv).astype(np.int32)).to(DEV)
        qs, ws_ = qd[p0:p1].contiguous(), wd[p0:p1].contiguous()
        i_r, s_r, _ = lidx.lidx_indexer_fwd_ranges(qs, kd, ws_, ks, ke, topk)
        assert torch.equal(i_r, full_i[:, p0:p1]) and torch.equal(s_r, full_s[:, p0:p1])
        dq_r, dk_r, dw_r = lidx.lidx_indexer_bwd_ranges(qs, kd, ws_, i_r, grad[:, p0:p1].contiguous(),
                                                        ks, ke)
        assert torch.equal(dq_r, fdq[p0:p1])
        # dw sums a row's key tiles in an order that follows the CTA's schedule:
        # equal up to fp32 reassociation
        assert torch.allclose(dw_r, fdw[p0:p1], rtol=1e-5, atol=1e-6 * fdw.abs().max().item())
        dk_sum += dk_r
    torch.cuda.synchronize()
    assert lidx.lidx_device_status() == 0
    err = (dk_sum - fdk).abs().max().item()
    assert err <= 1e-5 * fdk.abs().max().item(), err
