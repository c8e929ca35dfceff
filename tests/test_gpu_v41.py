"""GPU parity of the V4.1 bf16-rounded scorer (lidx_indexer_scores_v41)
against the CPU oracle: exact on integer-valued inputs; within one bf16 ulp on
>= 99.9% of visible entries otherwise, the rest within the bound of a head's
GEMM result rounding across a bf16 tie; -inf exactly where not visible."""

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_top_tcgen05_gb300 as lidx
import workloads
from parity import bf16_ulp_diff

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_attention_top_tcgen05_gb300 import build

    build.build()
    lidx.lib()
    yield
    assert lidx.lidx_device_status() == 0


def run(q, k, w, allowed, act="relu"):
    out = lidx.lidx_indexer_scores_v41(q.to(DEV), k.to(DEV), w.to(DEV), allowed.to(DEV), act=act)
    torch.cuda.synchronize()
    assert lidx.lidx_device_status() == 0
    return out.float().cpu().numpy()


def flip_bound(q, k, w, rows=None):
    """Per-entry bound on the score change when the fp32 GEMM result of one or
    two heads lies on the other side of a bf16 tie from the exact one (6 ulp of
    the largest weighted term), plus fp32 reduction error and final rounding."""
    B, S, H, D = q.shape
    r = np.arange(B * S) if rows is None else np.asarray(rows)
    qf = q.float().numpy().astype(np.float64).reshape(B * S, H, D)[r]
    wf = w.float().numpy().astype(np.float64).reshape(B * S, H)[r]
    kf = k.float().numpy().astype(np.float64)
    bidx = r // S
    out = np.empty((r.size, kf.shape[1]))
    ulp = lambda v: np.exp2(np.floor(np.log2(np.maximum(v, 1e-38))) - 7)
    for i in range(r.size):
        x = qf[i] @ kf[bidx[i]].T                 # [H, Skv]
        term = np.abs(x * wf[i][:, None])
        tot = np.abs((x * wf[i][:, None]).sum(0))
        out[i] = 6 * ulp(term.max(0)) + 2 * ulp(tot) + 64 * 2.0 ** -24 * term.sum(0)
    return out


def check(got, ref, allowed, exact=False, bound=None):
    al = allowed.numpy().reshape(got.shape).astype(bool)
    assert np.isneginf(got[~al]).all(), "invisible entries must be -inf"
    assert np.isfinite(got[al]).all()
    if exact:
        assert np.array_equal(got[al], ref[al])
    elif al.any():
        ulp = bf16_ulp_diff(got[al], ref[al])
        assert (ulp <= 1).mean() >= 0.999, (ulp <= 1).mean()
        if bound is not None and (ulp > 1).any():
            err = np.abs(got[al].astype(np.float64) - ref[al])
            bad = (ulp > 1) & (err > bound[al])
            assert not bad.any(), (err[bad][:5], bound[al][bad][:5])


@pytest.mark.parametrize("H,D", [(4, 16), (64, 128), (8, 32), (128, 64)])
def test_integer_inputs_bit_exact(H, D):
    B, S, Skv = 2, 160, 300
    q, k, w = workloads.integer_inputs(B, S, Skv, H, 16, seed=H)
    if D > 16:  # keep |q.k| small and every rounding exact: zero the extra dims
        q = torch.cat([q, torch.zeros(*q.shape[:-1], D - 16, dtype=q.dtype)], -1)
        k = torch.cat([k, torch.zeros(*k.shape[:-1], D - 16, dtype=k.dtype)], -1)
    q = q.permute(1, 0, 2, 3).contiguous()
    k = k.permute(1, 0, 2).contiguous()
    w = w.permute(1, 0, 2).contiguous().to(torch.bfloat16)
    allowed = torch.from_numpy(np.random.default_rng(H).random((B, S, Skv)) < 0.3)
    got = run(q, k, w, allowed).reshape(B * S, Skv)
    ref = oracle.scores_v41_rows(q, k, w, allowed)
    check(got, ref, allowed, exact=True)


def test_packed_documents_full_size_sampled():
    wl = workloads.WORKLOADS["v41_packed"]
    q, k, w, allowed = workloads.v41_inputs(wl, 0)
    got = run(q, k, w, allowed).reshape(wl.B * wl.S, wl.Skv)
    rows = workloads.sample_rows(wl.B, wl.S, 61, 5)
    ref = oracle.scores_v41_rows(q, k, w, allowed, rows=rows)
    check(got[rows], ref, allowed.reshape(wl.B * wl.S, wl.Skv)[rows],
          bound=flip_bound(q, k, w, rows=rows))
    # every masked entry of every row is -inf, every visible one finite
    al = allowed.numpy().reshape(wl.B * wl.S, wl.Skv)
    assert np.isneginf(got[~al]).all() and np.isfinite(got[al]).all()


@pytest.mark.parametrize("B,S,Skv,H,D,density", [
    (1, 300, 257, 64, 128, 0.5),   # ragged key tiles, Skv not a multiple of 4
    (2, 77, 1000, 16, 64, 0.05),
    (1, 64, 130, 1, 16, 0.9),
    (3, 40, 64, 32, 32, 1.0),
    # Skv % 16 == 0 takes the 16-byte visibility pass: a ragged last key tile, a key-tile
    # count that is not a multiple of four, blocks with no visible pair, none visible at all
    (2, 100, 400, 8, 64, 0.3),
    (1, 70, 208, 16, 32, 0.0005),
    (1, 33, 272, 4, 16, 0.0),
    (2, 300, 200, 2, 32, 0.4),     # 128 query rows a unit: flags read from global memory
])
def test_shapes_random_visibility(B, S, Skv, H, D, density):
    g = np.random.default_rng(S + Skv)
    q = workloads.to_bf16(g.standard_normal((B, S, H, D)).astype(np.float32) / np.sqrt(D))
    k = workloads.to_bf16(g.standard_normal((B, Skv, D)).astype(np.float32) / np.sqrt(D))
    w = workloads.to_bf16(g.standard_normal((B, S, H)).astype(np.float32) / np.sqrt(H))
    allowed = torch.from_numpy(g.random((B, S, Skv)) < density)
    bnd = flip_bound(q, k, w)
    got = run(q, k, w, allowed).reshape(B * S, Skv)
    check(got, oracle.scores_v41_rows(q, k, w, allowed), allowed, bound=bnd)
    gi = run(q, k, w, allowed, act="identity").reshape(B * S, Skv)
    check(gi, oracle.scores_v41_rows(q, k, w, allowed, act="identity"), allowed, bound=bnd)


@pytest.mark.parametrize("Skv", [9000, 8464])
def test_key_range_beyond_64_tiles(Skv):
    """A query tile whose visible pairs span more than 64 key tiles, with blocks
    of no visible pair inside the span on both sides of the 64th tile (9000: the
    word-load visibility pass; 8464: the 16-byte one)."""
    B, S, H, D = 1, 40, 16, 32
    g = np.random.default_rng(Skv)
    q = workloads.to_bf16(g.standard_normal((B, S, H, D)).astype(np.float32) / np.sqrt(D))
    k = workloads.to_bf16(g.standard_normal((B, Skv, D)).astype(np.float32) / np.sqrt(D))
    w = workloads.to_bf16(g.standard_normal((B, S, H)).astype(np.float32) / np.sqrt(H))
    ntk = (Skv + 127) // 128
    tiles = [1, 2, 40, 63, 64, 66, ntk - 1]
    al = np.zeros((B, S, Skv), dtype=bool)
    for t in tiles:
        lo, hi = t * 128, min(t * 128 + 128, Skv)
        al[:, :, lo:hi] = g.random((B, S, hi - lo)) < 0.3
    allowed = torch.from_numpy(al)
    got = run(q, k, w, allowed).reshape(B * S, Skv)
    check(got, oracle.scores_v41_rows(q, k, w, allowed), allowed, bound=flip_bound(q, k, w))


def test_all_false_and_all_true():
    g = np.random.default_rng(8)
    B, S, Skv, H, D = 1, 50, 200, 8, 32
    q = workloads.to_bf16(g.standard_normal((B, S, H, D)).astype(np.float32))
    k = workloads.to_bf16(g.standard_normal((B, Skv, D)).astype(np.float32))
    w = workloads.to_bf16(g.standard_normal((B, S, H)).astype(np.float32))
    none = torch.zeros(B, S, Skv, dtype=torch.bool)
    assert np.isneginf(run(q, k, w, none)).all()
    full = torch.ones(B, S, Skv, dtype=torch.bool)
    check(run(q, k, w, full).reshape(B * S, Skv), oracle.scores_v41_rows(q, k, w, full), full,
          bound=flip_bound(q, k, w))


# ------------------------------------------------------------------ V4.1 top-k
def run_topk(q, k, w, allowed, topk, act="relu"):
    sc, idx, tsc = lidx.lidx_indexer_topk_v41(q.to(DEV), k.to(DEV), w.to(DEV), allowed.to(DEV), topk,
                                              act=act)
    torch.cuda.synchronize()
    assert lidx.lidx_device_status() == 0
    return sc.float().cpu().numpy(), idx.cpu().numpy(), tsc.float().cpu().numpy()


def check_topk_on_own_scores(sc, idx, tsc, allowed, topk):
    """The selection equals the oracle's top-k of the kernel's own bf16 scores
    over the visible keys, bit for bit (scores are exact bf16 values)."""
    B, S, Skv = sc.shape
    al = allowed.numpy().reshape(B * S, Skv)
    oidx, osc = oracle.topk_masked_rows(sc.reshape(B * S, Skv).astype(np.float64), al, topk)
    assert np.array_equal(idx.reshape(B * S, topk), oidx)
    assert np.array_equal(tsc.reshape(B * S, topk).astype(np.float64), osc)


def test_topk_v41_packed_documents_full_size():
    """The V4.1 workload's shape (Skv 8192): bf16 scores as lidx_indexer_scores_v41,
    then the per-row top-512 over the visible keys."""
    wl = workloads.WORKLOADS["v41_packed"]
    q, k, w, allowed = workloads.v41_inputs(wl, 0)
    topk = wl.topk
    sc, idx, tsc = run_topk(q, k, w, allowed, topk)
    ref = run(q, k, w, allowed)
    assert np.array_equal(sc.reshape(ref.shape), ref)  # same scores as the scorer alone
    check_topk_on_own_scores(sc, idx, tsc, allowed, topk)
    n = allowed.numpy().reshape(wl.B * wl.S, wl.Skv).sum(1)
    assert (n > topk).any() and (n < topk).any()  # both selected and padded rows occur


@pytest.mark.parametrize("B,S,Skv,H,D,density,topk", [
    (1, 300, 257, 64, 128, 0.5, 100),   # rows not 16-byte aligned (bf16, Skv odd)
    (2, 77, 1000, 16, 64, 0.05, 64),
    (1, 64, 130, 1, 16, 0.9, 200),      # topk above every row's visible count
    (1, 33, 272, 4, 16, 0.0, 8),        # nothing visible
    (1, 40, 9000, 8, 32, 0.7, 4000),    # several candidate windows per row
    (1, 60, 512, 8, 32, 0.4, 100),      # one warp a row, 129 to 256 visible keys
    (1, 50, 1000, 16, 32, 0.6, 300),    # short span, too many visible keys for one warp
])
def test_topk_v41_shapes(B, S, Skv, H, D, density, topk):
    g = np.random.default_rng(S + Skv + topk)
    q = workloads.to_bf16(g.standard_normal((B, S, H, D)).astype(np.float32) / np.sqrt(D))
    k = workloads.to_bf16(g.standard_normal((B, Skv, D)).astype(np.float32) / np.sqrt(D))
    w = workloads.to_bf16(g.standard_normal((B, S, H)).astype(np.float32) / np.sqrt(H))
    allowed = torch.from_numpy(g.random((B, S, Skv)) < density)
    sc, idx, tsc = run_topk(q, k, w, allowed, topk)
    check_topk_on_own_scores(sc, idx, tsc, allowed, topk)
    # and the scores themselves are the oracle's within the scorer's tolerance
    check(sc.reshape(B * S, Skv), oracle.scores_v41_rows(q, k, w, allowed), allowed,
          bound=flip_bound(q, k, w))


def test_topk_v41_without_kept_scores_matches():
    g = np.random.default_rng(3)
    B, S, Skv, H, D, topk = 1, 128, 640, 32, 64, 50
    q = workloads.to_bf16(g.standard_normal((B, S, H, D)).astype(np.float32) / 8)
    k = workloads.to_bf16(g.standard_normal((B, Skv, D)).astype(np.float32) / 8)
    w = workloads.to_bf16(g.standard_normal((B, S, H)).astype(np.float32) / 4)
    allowed = torch.from_numpy(g.random((B, S, Skv)) < 0.4)
    sc, idx, tsc = run_topk(q, k, w, allowed, topk)
    none, idx2, tsc2 = lidx.lidx_indexer_topk_v41(q.to(DEV), k.to(DEV), w.to(DEV), allowed.to(DEV),
                                                  topk, keep_scores=False)
    assert none is None
    assert np.array_equal(idx2.cpu().numpy(), idx)
    assert np.array_equal(tsc2.float().cpu().numpy(), tsc)
