"""Repeated calls give identical bits.  The scoring kernels hand work between
warps through mbarrier rings (key tiles, accumulators, row buffers, V4.1
visibility records and flags) and the backward reduces in a fixed order, so a
race or a missed wait would show up as a call whose output differs from the
first one's.  Each workload runs many times at full size."""

import pytest
import torch

import sparse_attention_top_tcgen05_gb300 as lidx
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_attention_top_tcgen05_gb300 import build

    build.build()
    lidx.lib()
    yield
    assert lidx.lidx_device_status() == 0


def _same_every_time(fn, reps):
    first = [t.clone() for t in fn()]
    for _ in range(reps):
        again = fn()
        for a, b in zip(first, again):
            assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                               b.view(torch.uint8) if b.dtype == torch.bfloat16 else b)
    torch.cuda.synchronize()
    assert lidx.lidx_device_status() == 0


@pytest.mark.parametrize("name,S,reps", [("long_fused", 4096, 12), ("c4_fwd", 4096, 20), ("tiny", 256, 50)])
def test_fused_forward_repeats(name, S, reps):
    wl = workloads.WORKLOADS[name].with_(S=S)
    q, k, w = [t.to(DEV) for t in workloads.v4_inputs(wl, 1)]
    _same_every_time(lambda: lidx.lidx_indexer_fwd(q, k, w, wl.ratio, wl.topk)[:2], reps)


def test_v41_repeats():
    wl = workloads.WORKLOADS["v41_packed"]
    q, k, w, allowed = [t.to(DEV) for t in workloads.v41_inputs(wl, 1)]
    _same_every_time(lambda: (lidx.lidx_indexer_scores_v41(q, k, w, allowed),), 20)
    _same_every_time(lambda: lidx.lidx_indexer_topk_v41(q, k, w, allowed, wl.topk), 10)


def test_backward_repeats():
    wl = workloads.WORKLOADS["bwd"]
    q, k, w = [t.to(DEV) for t in workloads.v4_inputs(wl, 1)]
    idx, _, _ = lidx.lidx_indexer_fwd(q, k, w, wl.ratio, wl.topk)
    grad = workloads.grad_scores(wl.B, wl.S, wl.topk, 1).to(DEV)
    _same_every_time(lambda: lidx.lidx_indexer_bwd(q, k, w, idx, grad, wl.ratio), 8)
