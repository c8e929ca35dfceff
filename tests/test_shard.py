"""Sharding the path across ranks, on CPU with gloo (world size 2).

The indexer shards over query rows: each rank holds a contiguous shard of
query rows (their global positions fix the causal ranges) and all compressed
keys, as the context-parallel layout the V4.1 page describes ("keys ...
gathered across CP ranks before this call").  Rows are independent in the
forward, so the concatenated shards must equal the unsharded result exactly;
in the backward dq and dw stay local and dk is the sum of the ranks' partial
dk.  The benchmark's max-over-ranks timing helper is checked on the same
process group."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _case():
    import workloads

    wl = workloads.WORKLOADS["tiny"].with_(S=64, Skv=16, H=4, D=16, topk=6)
    q, k, w = workloads.v4_inputs(wl, 7)
    return wl, q, k, w


def _worker(rank, world, port, out_dir):
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    import oracle
    import workloads

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    oracle.set_threads(1)
    wl, q, k, w = _case()
    S = wl.S
    shard = np.arange(rank * S // world, (rank + 1) * S // world)  # global query rows
    idx, sc, _ = oracle.indexer_fwd_rows(q, k, w, wl.ratio, wl.topk, rows=shard)
    gi = [torch.zeros(len(shard), wl.topk, dtype=torch.int32) for _ in range(world)]
    gs = [torch.zeros(len(shard), wl.topk, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(gi, torch.from_numpy(idx))
    dist.all_gather(gs, torch.from_numpy(sc))
    # backward: this rank's rows only, dk summed across ranks
    ks, ke = oracle.causal_ranges(S, wl.Skv, wl.ratio)
    sel = workloads.random_selection(1, S, wl.Skv, wl.topk, ke - ks, 3).numpy()
    grad = workloads.grad_scores(1, S, wl.topk, 3).numpy()
    mine = sel.copy()
    mask = np.ones(S, bool)
    mask[shard] = False
    mine[:, mask] = -1
    dq, dk, dw, *_ = oracle.bwd(q, k, w, mine, grad, ks, ke, slack=False)
    dkt = torch.from_numpy(dk)
    dist.all_reduce(dkt)
    t = bench.max_over_ranks(float(rank + 1), world)
    if rank == 0:
        np.savez(os.path.join(out_dir, "r0.npz"), idx=torch.cat(gi).numpy(), sc=torch.cat(gs).numpy(),
                 dk=dkt.numpy(), maxt=t)
    np.savez(os.path.join(out_dir, f"rows{rank}.npz"), dq=dq[shard], dw=dw[shard], shard=shard)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_query_sharding(tmp_path):
    import oracle
    import workloads

    oracle.build()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    r0 = np.load(tmp_path / "r0.npz")
    wl, q, k, w = _case()
    idx, sc, _ = oracle.indexer_fwd_rows(q, k, w, wl.ratio, wl.topk)
    assert np.array_equal(r0["idx"], idx)
    assert np.array_equal(r0["sc"], sc)
    ks, ke = oracle.causal_ranges(wl.S, wl.Skv, wl.ratio)
    sel = workloads.random_selection(1, wl.S, wl.Skv, wl.topk, ke - ks, 3).numpy()
    grad = workloads.grad_scores(1, wl.S, wl.topk, 3).numpy()
    dq, dk, dw, *_ = oracle.bwd(q, k, w, sel, grad, ks, ke, slack=False)
    np.testing.assert_allclose(r0["dk"], dk, rtol=1e-12, atol=1e-12)
    for r in range(2):
        part = np.load(tmp_path / f"rows{r}.npz")
        assert np.array_equal(part["dq"], dq[part["shard"]])
        assert np.array_equal(part["dw"], dw[part["shard"]])
    assert float(r0["maxt"]) == 2.0  # max over ranks of (rank + 1)
