"""Failure detection on the GPU without a fault: every pipeline wait in the
scoring kernel gives up after a time limit, records LIDX_ERR_DEVICE_TIMEOUT in
the status word and winds the kernel down.  Here a test switch stops the TMA
producer, so no load ever lands and every wait runs out; the launch ends on
its own, the host reads the status, and the next normal call is correct."""

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_top_tcgen05_gb300 as lidx
import workloads

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
