"""The workspace-free fused forward (lidx_indexer_fwd_noalloc) must give what
the workspace-taking entry point (lidx_indexer_fwd) gives.

It exists for callers that cannot allocate device memory -- code running
inside an allocator callback, in a process whose device memory another
framework has reserved, or in a plug-in that only receives input and output
pointers -- so it takes its scratch from an array inside the library.  This
file is collected last so that a stop-at-first-failure run has already run
every other test if this one fails."""

import ctypes as C

import numpy as np
import pytest
import torch

import sparse_attention_top_tcgen05_gb300 as lidx
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def L():
    from sparse_attention_top_tcgen05_gb300 import build

    build.build()
    return lidx.lib()


def _inputs(seed, wl):
    return [t.to(DEV) for t in workloads.v4_inputs(wl, seed)]


def _noalloc(L, q, k, w, ratio, topk):
    """One call through the C ABI with caller-owned outputs only."""
    S, B, H, D = q.shape
    Skv = k.shape[0]
    idx = torch.full((B, S, topk), 7, dtype=torch.int32, device=DEV)
    sc = torch.full((B, S, topk), 7.0, dtype=torch.float32, device=DEV)
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.lidx_indexer_fwd_noalloc(C.c_void_p(q.data_ptr()), C.c_void_p(k.data_ptr()),
                                    C.c_void_p(w.data_ptr()), B, S, Skv, H, D, ratio, topk, 0,
                                    C.c_void_p(idx.data_ptr()), C.c_void_p(sc.data_ptr()), stream)
    return rc, idx, sc


def test_noalloc_matches_workspace_entry_point_twice(L):
    wl = workloads.WORKLOADS["c4_fwd"]
    runs = []
    for seed in (0, 1):  # two calls in a row, different inputs: no stale scratch
        q, k, w = _inputs(seed, wl)
        rc, idx, sc = _noalloc(L, q, k, w, wl.ratio, wl.topk)
        assert rc == 0, lidx.lidx_status_string(rc)
        runs.append((q, k, w, idx, sc))
    torch.cuda.synchronize()
    assert lidx.lidx_device_status() == 0
    for q, k, w, idx, sc in runs:
        ridx, rsc, _ = lidx.lidx_indexer_fwd(q, k, w, wl.ratio, wl.topk)
        torch.cuda.synchronize()
        # same kernel and arithmetic: identical selections and scores
        assert np.array_equal(idx.cpu().numpy(), ridx.cpu().numpy())
        assert np.array_equal(sc.cpu().numpy(), rsc.cpu().numpy())
    assert not np.array_equal(runs[0][3].cpu().numpy(), runs[1][3].cpu().numpy())


def test_noalloc_rejects_sizes_beyond_its_array(L):
    limit = L.lidx_noalloc_scratch_bytes()
    assert limit == 24 << 20
    wl = workloads.WORKLOADS["tiny"].with_(H=8, D=32, S=64, Skv=4096)  # 32 queries per tile
    need = lidx.lidx_workspace_bytes(lidx.OP_INDEXER_FWD, wl.B, wl.S, wl.Skv, wl.H, wl.D, 16)
    assert need > limit
    q = torch.zeros(wl.S, 1, wl.H, wl.D, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(wl.Skv, 1, wl.D, dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(wl.S, 1, wl.H, device=DEV)
    rc, idx, sc = _noalloc(L, q, k, w, 4, 16)
    assert rc == 5  # LIDX_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert (idx == 7).all()


def test_noalloc_checks_arguments_before_its_size_limit(L):
    """A bad shape is reported as a shape error even when the call would also
    be too large for the array."""
    q = torch.zeros(64, 1, 8, 32, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(4096, 1, 32, dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(64, 1, 8, device=DEV)
    idx = torch.empty(1, 64, 16, dtype=torch.int32, device=DEV)
    sc = torch.empty(1, 64, 16, device=DEV)
    P = lambda t: C.c_void_p(t.data_ptr())
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    # D = 24 is not a multiple of 16
    rc = L.lidx_indexer_fwd_noalloc(P(q), P(k), P(w), 1, 64, 4096, 8, 24, 4, 16, 0, P(idx), P(sc), stream)
    assert rc == 2  # LIDX_ERR_SHAPE
    rc = L.lidx_indexer_fwd_noalloc(P(q), P(k), P(w), 1, 64, 4096, 8, 32, 0, 16, 0, P(idx), P(sc), stream)
    assert rc == 2  # compress_ratio 0


def test_noalloc_at_the_edge_of_its_array(L):
    """The largest key count whose scratch fits the array on this device runs
    and matches the workspace entry point; one key more is rejected."""
    limit = L.lidx_noalloc_scratch_bytes()
    H, D = 8, 32
    fits = [s for s in range(128, 4097, 128)
            if lidx.lidx_workspace_bytes(lidx.OP_INDEXER_FWD, 1, 1, s, H, D, 16) <= limit]
    Skv = max(fits)
    assert lidx.lidx_workspace_bytes(lidx.OP_INDEXER_FWD, 1, 1, Skv + 1, H, D, 16) > limit
    wl = workloads.WORKLOADS["tiny"].with_(S=Skv + 60, Skv=Skv, H=H, D=D, ratio=1, topk=40)
    q, k, w = _inputs(5, wl)
    rc, idx, sc = _noalloc(L, q, k, w, 1, wl.topk)
    assert rc == 0, lidx.lidx_status_string(rc)
    ridx, rsc, _ = lidx.lidx_indexer_fwd(q, k, w, 1, wl.topk)
    torch.cuda.synchronize()
    assert torch.equal(idx, ridx) and torch.equal(sc, rsc)
    wl2 = wl.with_(Skv=Skv + 1)
    q2, k2, w2 = _inputs(6, wl2)
    rc, idx2, _ = _noalloc(L, q2, k2, w2, 1, wl2.topk)
    assert rc == 5  # LIDX_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert (idx2 == 7).all()
