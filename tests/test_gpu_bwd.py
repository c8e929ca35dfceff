"""GPU parity of the backward (lidx_indexer_bwd) against the CPU oracle.

Tolerance per tensor: 1e-3 relative or 1e-3*max|ref| absolute, widened per
element by the oracle's slack for pairs whose ReLU decision lies within fp32
accumulation error.  The backward uses no atomics on its outputs, so two runs
must agree bit for bit; bf16 outputs are the fp32 results rounded once."""

import numpy as np
import pytest
import torch

import oracle
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


def close(got, ref, slack, name):
    got = np.asarray(got, np.float64)
    tol = 1e-3 * max(np.abs(ref).max(), 1e-30)
    err = np.abs(got - ref)
    ok = (err <= tol + slack) | (err <= 1e-3 * np.abs(ref) + slack)
    assert ok.all(), f"{name}: max err {err.max():.3e}, tol {tol:.3e}, at {np.argwhere(~ok)[:3]}"


def run_case(q, k, w, idx, grad, ratio, act="relu"):
    S, B, H, D = q.shape
    Skv = k.shape[0]
    dq, dk, dw = lidx.lidx_indexer_bwd(q.to(DEV), k.to(DEV), w.to(DEV), torch.as_tensor(idx).to(DEV),
                                       torch.as_tensor(grad).to(DEV), ratio, act=act)
    torch.cuda.synchronize()
    assert lidx.lidx_device_status() == 0
    ks, ke = oracle.causal_ranges(S, Skv, ratio)
    rq, rk, rw, sq, sk, sw = oracle.bwd(q, k, w, idx, grad, ks, ke, act=act)
    close(dq.cpu().numpy(), rq, sq, "dq")
    close(dk.cpu().numpy(), rk, sk, "dk")
    close(dw.cpu().numpy(), rw, sw, "dw")


def selection(B, S, Skv, ratio, topk, seed):
    ks, ke = oracle.causal_ranges(S, Skv, ratio)
    return workloads.random_selection(B, S, Skv, topk, ke - ks, seed).numpy()


@pytest.mark.parametrize("B,S,H,D,Skv,ratio,topk", [
    (2, 300, 8, 32, 80, 4, 24),
    (1, 257, 64, 128, 200, 1, 100),
    (3, 100, 128, 64, 30, 2, 40),     # topk > visible keys: padding slots
    (1, 129, 1, 16, 129, 1, 7),
    (1, 200, 16, 64, 300, 2, 50),     # heads below 32: one grad per column in the key-major pass
    (2, 150, 32, 128, 260, 1, 90),
    (1, 700, 4, 48, 650, 1, 300),     # index_dim not a multiple of 64
    (1, 1100, 8, 32, 1100, 1, 1100),  # more than 1024 slots a row: the scatter reads them in place
])
def test_random_selection(B, S, H, D, Skv, ratio, topk):
    g = np.random.default_rng(S + H)
    q = workloads.to_bf16(g.standard_normal((S, B, H, D)).astype(np.float32) / np.sqrt(D))
    k = workloads.to_bf16(g.standard_normal((Skv, B, D)).astype(np.float32) / np.sqrt(D))
    w = torch.from_numpy((g.standard_normal((S, B, H)) / np.sqrt(H)).astype(np.float32))
    idx = selection(B, S, Skv, ratio, topk, 1)
    grad = workloads.grad_scores(B, S, topk, 1).numpy()
    run_case(q, k, w, idx, grad, ratio)
    run_case(q, k, w, idx, grad, ratio, act="identity")


def test_invisible_and_padding_slots_carry_no_gradient():
    g = np.random.default_rng(5)
    B, S, H, D, Skv, ratio, topk = 1, 64, 8, 32, 16, 4, 6
    q = workloads.to_bf16(g.standard_normal((S, B, H, D)).astype(np.float32))
    k = workloads.to_bf16(g.standard_normal((Skv, B, D)).astype(np.float32))
    w = torch.from_numpy(g.standard_normal((S, B, H)).astype(np.float32))
    idx = g.integers(-3, Skv + 3, (B, S, topk)).astype(np.int32)  # many outside the causal range
    grad = g.standard_normal((B, S, topk)).astype(np.float32)
    run_case(q, k, w, idx, grad, ratio)


def test_backward_workload_sampled_rows():
    """Full-size backward workload in the benchmark's launch configuration; the
    selection is kept on a strided sample of rows (others all -1) so that the
    fp64 oracle covers every output exactly, dk included."""
    wl = workloads.WORKLOADS["bwd"]
    ks, ke = oracle.causal_ranges(wl.S, wl.Skv, wl.ratio)
    q, k, w, idx, grad = workloads.bwd_inputs(wl, ke - ks, 0)
    idx = idx.numpy()
    keep = np.zeros(wl.S, bool)
    keep[workloads.sample_rows(1, wl.S, 97, 11)] = True
    idx[:, ~keep] = -1
    run_case(q, k, w, idx, grad.numpy(), wl.ratio)


def test_deterministic_and_bf16_outputs():
    """Two runs give identical bits; grad_dtype bf16 returns the fp32 results
    rounded to nearest-even once."""
    wl = workloads.WORKLOADS["bwd"].with_(S=2048, Skv=512, topk=256)
    ks, ke = oracle.causal_ranges(wl.S, wl.Skv, wl.ratio)
    q, k, w, idx, grad = workloads.bwd_inputs(wl, ke - ks, 3)
    args = [t.to(DEV) for t in (q, k, w, idx, grad)]
    a = lidx.lidx_indexer_bwd(*args, wl.ratio)
    b = lidx.lidx_indexer_bwd(*args, wl.ratio)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    c = lidx.lidx_indexer_bwd(*args, wl.ratio, grad_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert lidx.lidx_device_status() == 0
    assert c[0].dtype == torch.bfloat16 and c[1].dtype == torch.bfloat16
    assert torch.equal(c[0], a[0].to(torch.bfloat16)) and torch.equal(c[1], a[1].to(torch.bfloat16))
    assert torch.equal(c[2], a[2])
