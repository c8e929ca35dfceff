"""Failure detection on the GPU without a fault: every pipeline wait in the
scoring kernels and the backward gives up after a time limit, records
LIDX_ERR_DEVICE_TIMEOUT in the status word and winds the kernel down.  Here a
test switch stops the TMA producer, so no load ever lands and every wait runs
out; the launch ends on its own, the host reads the status, and the next normal
call is correct."""

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_top_tcgen05_gb300 as lidx
import workloads
from parity import bf16_ulp_diff

pytestmark = pytest.mark.gpu
DEV = "cuda"
LIDX_ERR_DEVICE_TIMEOUT = 7


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_attention_top_tcgen05_gb300 import build

    build.build()
    lidx.lib()
    yield
    lidx.lidx_debug_stall_producer(False)
    lidx.lidx_set_wait_limit_ns(0)


def test_stalled_pipeline_times_out_and_the_next_call_is_correct():
    wl = workloads.WORKLOADS["tiny"]
    q, k, w = workloads.v4_inputs(wl, 0)
    qd, kd, wd = q.to(DEV), k.to(DEV), w.to(DEV)
    assert lidx.lidx_device_status() == 0
    old = lidx.lidx_set_wait_limit_ns(2_000_000)  # 2 ms
    lidx.lidx_debug_stall_producer(True)
    try:
        lidx.lidx_indexer_fwd(qd, kd, wd, wl.ratio, wl.topk)  # fused: every role waits
        lidx.lidx_indexer_fwd(qd, kd, wd, wl.ratio, wl.topk, materialise_logits=True)
        assert lidx.lidx_device_status() == LIDX_ERR_DEVICE_TIMEOUT
        assert lidx.lidx_device_status() == 0  # reading clears it
    finally:
        lidx.lidx_debug_stall_producer(False)
        lidx.lidx_set_wait_limit_ns(old)
    idx, sc, lg = lidx.lidx_indexer_fwd(qd, kd, wd, wl.ratio, wl.topk, materialise_logits=True)
    torch.cuda.synchronize()
    assert lidx.lidx_device_status() == 0
    oidx, osc, olg = oracle.indexer_fwd_rows(q, k, w, wl.ratio, wl.topk)
    glg = lg.cpu().numpy().reshape(wl.S, wl.Skv)
    fin = np.isfinite(olg)
    assert np.array_equal(np.isfinite(glg), fin)
    assert np.abs(glg[fin] - olg[fin]).max() <= 1e-3 * np.abs(olg[fin]).max()
    ks, ke = oracle.causal_ranges(wl.S, wl.Skv, wl.ratio)
    ridx, _ = oracle.topk_rows(glg.astype(np.float64), wl.S, ks, ke, wl.topk, np.arange(wl.S))
    assert np.array_equal(idx.cpu().numpy().reshape(wl.S, wl.topk), ridx)


class _Stalled:
    """The producer switched off and a 2 ms wait limit, for one block."""

    def __enter__(self):
        assert lidx.lidx_device_status() == 0
        self.old = lidx.lidx_set_wait_limit_ns(2_000_000)
        lidx.lidx_debug_stall_producer(True)

    def __exit__(self, *exc):
        lidx.lidx_debug_stall_producer(False)
        lidx.lidx_set_wait_limit_ns(self.old)


def test_v41_stall_times_out_and_the_next_call_is_correct():
    """More than four query tiles per CTA, so the visibility warps also wait for a
    record slot that no consumer frees, and give up."""
    B, S, Skv, H, D = 1, 4096, 256, 64, 32
    g = np.random.default_rng(41)
    q = workloads.to_bf16(g.standard_normal((B, S, H, D)).astype(np.float32) / np.sqrt(D))
    k = workloads.to_bf16(g.standard_normal((B, Skv, D)).astype(np.float32) / np.sqrt(D))
    w = workloads.to_bf16(g.standard_normal((B, S, H)).astype(np.float32) / np.sqrt(H))
    allowed = torch.from_numpy(g.random((B, S, Skv)) < 0.3)
    qd, kd, wd, ad = q.to(DEV), k.to(DEV), w.to(DEV), allowed.to(DEV)
    with _Stalled():
        lidx.lidx_indexer_scores_v41(qd, kd, wd, ad)
        assert lidx.lidx_device_status() == LIDX_ERR_DEVICE_TIMEOUT
    got = lidx.lidx_indexer_scores_v41(qd, kd, wd, ad).float().cpu().numpy().reshape(B * S, Skv)
    assert lidx.lidx_device_status() == 0
    ref = oracle.scores_v41_rows(q, k, w, allowed)
    al = allowed.numpy().reshape(B * S, Skv)
    assert np.isneginf(got[~al]).all()
    assert (bf16_ulp_diff(got[al], ref[al]) <= 1).mean() >= 0.999


def test_backward_stall_times_out_and_the_next_call_is_correct():
    B, S, H, D, Skv, ratio, topk = 1, 300, 8, 32, 80, 4, 24
    wl = workloads.WORKLOADS["tiny"].with_(B=B, S=S, H=H, D=D, Skv=Skv, topk=topk)
    q, k, w = workloads.v4_inputs(wl, 5)
    ks, ke = oracle.causal_ranges(S, Skv, ratio)
    idx = workloads.random_selection(B, S, Skv, topk, ke - ks, 5).numpy()
    grad = workloads.grad_scores(B, S, topk, 5)
    args = (q.to(DEV), k.to(DEV), w.to(DEV), torch.as_tensor(idx).to(DEV), grad.to(DEV), ratio)
    with _Stalled():
        lidx.lidx_indexer_bwd(*args)
        assert lidx.lidx_device_status() == LIDX_ERR_DEVICE_TIMEOUT
    dq, dk, dw = lidx.lidx_indexer_bwd(*args)
    torch.cuda.synchronize()
    assert lidx.lidx_device_status() == 0
    rq, rk, rw, sq, sk, sw = oracle.bwd(q, k, w, idx, grad.numpy(), ks, ke)
    for got, ref, sl in ((dq, rq, sq), (dk, rk, sk), (dw, rw, sw)):
        got = got.cpu().numpy().astype(np.float64)
        err = np.abs(got - ref)
        assert (err <= 1e-3 * max(np.abs(ref).max(), 1e-30) + sl).all()
