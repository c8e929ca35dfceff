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
