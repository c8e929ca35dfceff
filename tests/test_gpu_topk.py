"""GPU parity of the standalone selection (lidx_topk_rows) and the gather
(lidx_extract_topk_scores): both must equal the oracle bit for bit on the same
fp32 inputs, including adversarial rows (ties, outliers, ranges)."""

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_top_tcgen05_gb300 as lidx

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_attention_top_tcgen05_gb300 import build

    build.build()
    lidx.lib()
    yield
    assert lidx.lidx_device_status() == 0


def rows_case(kind, S, Skv, seed):
    g = np.random.default_rng(seed)
    if kind == "normal":
        x = g.standard_normal((S, Skv)).astype(np.float32)
    elif kind == "ties":      # few distinct values: many exact ties
        x = g.integers(-3, 4, (S, Skv)).astype(np.float32) * 0.5
    elif kind == "outlier":   # one huge value, the rest in a narrow band
        x = (g.standard_normal((S, Skv)) * 1e-3).astype(np.float32)
        x[:, 7 % Skv] = 1e30
    elif kind == "const":
        x = np.full((S, Skv), 2.5, np.float32)
    elif kind == "heavy":     # heavy tail
        x = (g.standard_cauchy((S, Skv)) * 10).astype(np.float32)
    elif kind == "tiny_range":  # values differing in the last bits only
        x = (1.0 + g.integers(0, 64, (S, Skv)) * 2.0 ** -23).astype(np.float32)
    elif kind == "zero_pad":  # keys past a short prefix are zero: most scores exactly 0
        x = g.standard_normal((S, Skv)).astype(np.float32)
        x[:, Skv // 8:] = 0.0
    elif kind == "two_values":  # two values only: buckets larger than a shared-memory window
        x = np.where(g.random((S, Skv)) < 0.5, 1.0, -2.0).astype(np.float32)
    elif kind == "band":  # one outlier; the rest distinct values in a narrow band
        x = (1.0 + g.random((S, Skv)) * 1e-4).astype(np.float32)
        x[:, 3 % Skv] = -1e30
    else:
        raise ValueError(kind)
    return x


@pytest.mark.parametrize("kind", ["normal", "ties", "outlier", "const", "heavy", "tiny_range"])
@pytest.mark.parametrize("S,Skv,ratio,topk", [(300, 1024, 1, 100), (1000, 4096, 4, 2048), (64, 50, 1, 64)])
def test_topk_rows_bit_exact(kind, S, Skv, ratio, topk):
    x = rows_case(kind, S, Skv, S + Skv)
    lg = torch.from_numpy(x).to(DEV)
    idx, sc = lidx.lidx_topk_rows(lg.reshape(1, S, Skv), topk, compress_ratio=ratio)
    torch.cuda.synchronize()
    ks, ke = oracle.causal_ranges(S, Skv, ratio)
    oidx, osc = oracle.topk_rows(x.astype(np.float64), S, ks, ke, topk, np.arange(S))
    assert np.array_equal(idx.cpu().numpy().reshape(S, topk), oidx)
    assert np.array_equal(sc.cpu().numpy().reshape(S, topk).astype(np.float64), osc)


@pytest.mark.parametrize("kind", ["normal", "ties", "const", "outlier", "heavy", "tiny_range",
                                  "zero_pad", "two_values", "band"])
@pytest.mark.parametrize("S,Skv,topk", [(40, 8192, 2048), (24, 16384, 6000), (9, 20000, 19000)])
def test_topk_rows_long_rows_bit_exact(kind, S, Skv, topk):
    """Rows longer than one shared-memory window of candidates (several
    windows, refined buckets, all-equal items) select exactly what the oracle
    selects.  Explicit ranges: the first half of the rows grow from 1 key to
    the full width, the rest see the full width."""
    x = rows_case(kind, S, Skv, S * 7 + Skv)
    lg = torch.from_numpy(x).to(DEV)
    ks = np.zeros(S, np.int32)
    ke = np.full(S, Skv, np.int32)
    ke[: S // 2] = np.linspace(1, Skv, S // 2).astype(np.int32)
    idx, sc = lidx.lidx_topk_rows(lg.reshape(1, S, Skv), topk, ks=torch.from_numpy(ks).to(DEV),
                                  ke=torch.from_numpy(ke).to(DEV))
    torch.cuda.synchronize()
    assert lidx.lidx_device_status() == 0
    oidx, osc = oracle.topk_rows(x.astype(np.float64), S, ks, ke, topk, np.arange(S))
    assert np.array_equal(idx.cpu().numpy().reshape(S, topk), oidx)
    assert np.array_equal(sc.cpu().numpy().reshape(S, topk).astype(np.float64), osc)


def test_topk_rows_explicit_ranges_and_batches():
    g = np.random.default_rng(1)
    B, S, Skv, topk = 3, 200, 700, 64
    x = g.standard_normal((B, S, Skv)).astype(np.float32)
    ks = g.integers(-10, Skv, S).astype(np.int32)
    ke = (ks + g.integers(-5, 400, S)).astype(np.int32)
    idx, sc = lidx.lidx_topk_rows(torch.from_numpy(x).to(DEV), topk,
                                  ks=torch.from_numpy(ks).to(DEV), ke=torch.from_numpy(ke).to(DEV))
    oidx, osc = oracle.topk_rows(x.reshape(B * S, Skv).astype(np.float64), S, ks, ke, topk,
                                 np.arange(B * S))
    assert np.array_equal(idx.cpu().numpy().reshape(B * S, topk), oidx)
    assert np.array_equal(sc.cpu().numpy().reshape(B * S, topk).astype(np.float64), osc)


def test_extract_matches_oracle_gather():
    g = np.random.default_rng(2)
    B, S, Skv, topk = 2, 100, 333, 40
    x = g.standard_normal((B, S, Skv)).astype(np.float32)
    ridx = g.integers(-5, Skv + 5, (B, S, topk)).astype(np.int32)
    out = lidx.lidx_extract_topk_scores(torch.from_numpy(x).to(DEV), torch.from_numpy(ridx).to(DEV))
    ref = oracle.extract_rows(x.reshape(B * S, Skv), ridx.reshape(B * S, topk))
    assert np.array_equal(out.cpu().numpy().reshape(B * S, topk).astype(np.float64), ref)
