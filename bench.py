"""Benchmark of the lightning-indexer hot path on one GB300 (or N replicas).

Headline: the fused long-context V4 forward (score + causal mask + top-k,
logits never written) at B=2, S=16384, H=64, D=128, compress_ratio 4
(Skv=4096), topk=2048, bf16 inputs, fp32 accumulation.

  value  = valid-pair TFLOP/s = (visible causal pairs x 2*H*D) / step time,
           inputs resident in HBM (q alone is 537 MB, larger than the 129 MB L2)
  e2e    = the same metric through the C ABI with host buffers: pinned
           host->device copy of q, k, w and device->host copy of indices and
           scores inside the timed region, every step; consecutive steps overlap
           on three streams (copy in, compute, copy out) with two buffer sets
  roofline: the scoring kernel against the measured dense bf16 peak
  cpu_baseline: the CPU oracle on a strided sample of the same rows

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun each rank runs one replica; rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SCORE_SRC = ["sparse_attention_top_tcgen05_gb300/csrc/score_fwd.cuh",
             "sparse_attention_top_tcgen05_gb300/csrc/score_fwd.cu",
             "sparse_attention_top_tcgen05_gb300/csrc/score_fwd_v4_fused.cu",
             "sparse_attention_top_tcgen05_gb300/csrc/topk.cuh",
             "sparse_attention_top_tcgen05_gb300/csrc/ptx.cuh"]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def src_hash(paths):
    h = hashlib.sha256()
    for rel in paths:
        h.update(open(os.path.join(ROOT, rel), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key, paths):
    """dram bytes per launch from a committed ncu summary, if it was taken on
    the current source of the kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_key)
    if not d or d.get("src_hash") != src_hash(paths):
        return None
    return d.get("dram_bytes_per_launch")


def visible_pairs(S, Skv, ratio, B):
    s = np.arange(S, dtype=np.int64)
    return int(np.minimum((s + 1) // ratio, Skv).sum()) * B


class Clocks:
    """nvidia-smi sampler running while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle
_CPU_INPUTS = {}


def cpu_oracle_sample(wl, stride, seed=0):
    """Time the oracle (as it stands) on every `stride`-th row of the workload."""
    import oracle

    key = (wl.name, wl.B, wl.S, wl.Skv, seed)
    if key not in _CPU_INPUTS:
        _CPU_INPUTS.clear()
        _CPU_INPUTS[key] = workloads.v4_inputs(wl, seed)
    q, k, w = _CPU_INPUTS[key]
    rows = workloads.sample_rows(wl.B, wl.S, stride, 0)
    ks, ke = oracle.causal_ranges(wl.S, wl.Skv, wl.ratio)
    pairs = int(sum(ke[r % wl.S] - ks[r % wl.S] for r in rows))
    t0 = time.perf_counter()
    oracle.indexer_fwd_rows(q, k, w, wl.ratio, wl.topk, rows=rows)
    dt = time.perf_counter() - t0
    flops = pairs * 2.0 * wl.H * wl.D
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.get_threads(),
            "kind": "oracle", "rows_per_s": len(rows) / dt, "seconds": dt,
            "sample": f"{len(rows)} query rows (every {stride}th row of each batch plus the last), "
                      f"{pairs} visible pairs, full fp64 logits + top-k per row"}


def run_reference(args, wl, world, rank):
    if rank != 0:
        return
    steps = []
    stride = 64
    for _ in range(args.warmup):
        cpu_oracle_sample(wl, stride * 4)
    for _ in range(args.steps):
        steps.append(cpu_oracle_sample(wl, stride))
    v = statistics.median(s["value"] for s in steps)
    cb = dict(steps[0])
    cb["value"] = v
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.median(s["seconds"] for s in steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(wl, 1),
            "cpu_baseline": cb,
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


METRIC = "indexer valid-pair TFLOP/s and query-rows/s incl. top-k; % of GB300 BF16 peak"


WORKLOAD_DESC = {
    "tiny": "V4 score+causal mask+top-k, logits materialised",
    "c4_fwd": "V4 C4-layer score+causal mask, logits materialised, then top-k",
    "long_fused": "V4 fused score+causal mask+top-k, logits not materialised",
    "bwd": "V4 fused score+causal mask+top-k at the backward workload's shape",
}


def config_of(wl, n):
    desc = WORKLOAD_DESC.get(wl.name, "V4 fused score+causal mask+top-k")
    q_mb = wl.B * wl.S * wl.H * wl.D * 2 / 1e6
    return {"workload": f"{wl.name}: {desc}",
            "B": wl.B, "S": wl.S, "H": wl.H, "D": wl.D, "Skv": wl.Skv,
            "compress_ratio": wl.ratio, "topk": wl.topk, "act": "relu",
            "inputs": "bf16 q,k ~N(0,1/D); fp32 w ~N(0,1/H); seed 0",
            "l2": (f"inputs larger than L2 (q = {q_mb:.0f} MB > 129 MB), no flush" if q_mb > 129
                   else f"q = {q_mb:.0f} MB fits in L2 (129 MB): a profiling size, not the workload"),
            "parallelism": f"replicas x{n}"}


# ------------------------------------------------------------------- GPU arm
def time_steps(fn, steps, stream):
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / steps


def _median_ms(fn, stream, reps, flush=None):
    """Median device time of one call.  The L2 flush (a 256 MB write, tens of
    microseconds on the device) is enqueued on the same stream first, so that
    the call's launches are queued behind it and the events bracket device work
    only, not the host's launch latency."""
    ts = []
    for _ in range(reps):
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            if flush is not None:
                flush.zero_()
            start.record(stream)
            fn()
            end.record(stream)
        end.synchronize()
        ts.append(start.elapsed_time(end))
    return statistics.median(ts)


def selection_rows(kind, rows, Skv, seed=0):
    """Adversarial score rows for the selection timing (fp32 [rows, Skv])."""
    g = np.random.default_rng(seed)
    if kind == "normal":
        x = g.standard_normal((rows, Skv))
    elif kind == "ties":        # seven distinct values
        x = g.integers(-3, 4, (rows, Skv)) * 0.5
    elif kind == "const":
        x = np.full((rows, Skv), 2.5)
    elif kind == "zero_pad":    # most keys score exactly 0
        x = g.standard_normal((rows, Skv))
        x[:, Skv // 8:] = 0.0
    elif kind == "two_values":
        x = np.where(g.random((rows, Skv)) < 0.5, 1.0, -2.0)
    else:
        raise ValueError(kind)
    return torch.from_numpy(x.astype(np.float32))


def side_workloads(lidx, pk, names=None):
    """Short measurements of the other workloads' kernels (not the headline);
    ``names`` picks a subset of tiny, c4_fwd, v41_packed, selection, bwd."""
    out = {}
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")

    def _tiny():
        # tiny workload: latency of one call (logits materialised, then top-k)
        wl = workloads.WORKLOADS["tiny"]
        q, k, w = [t.cuda() for t in workloads.v4_inputs(wl, 0)]
        idx = torch.empty(wl.B, wl.S, wl.topk, dtype=torch.int32, device="cuda")
        sc = torch.empty_like(idx, dtype=torch.float32)
        lg = torch.empty(wl.B, wl.S, wl.Skv, dtype=torch.float32, device="cuda")
        fn = lambda: lidx.lidx_indexer_fwd(q, k, w, wl.ratio, wl.topk, materialise_logits=True,
                                           out=(idx, sc, lg))
        for _ in range(10):
            fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(200):
            fn()
        torch.cuda.synchronize()
        host_us = (time.perf_counter() - t0) / 200 * 1e6
        # device time of one call: 20 calls captured in a CUDA graph and replayed, so
        # that host launch latency is out of the measurement
        dev_us = None
        try:
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                fn()
                torch.cuda.synchronize()
                with torch.cuda.graph(g, stream=side):
                    for _ in range(20):
                        fn()
            torch.cuda.synchronize()
            for _ in range(3):
                g.replay()
            dev_us = 1e3 * time_steps(g.replay, 50, torch.cuda.current_stream()) / 20
        except RuntimeError as e:  # capture refused: report the back-to-back rate only
            dev_us = f"unavailable: {e}"
        out["tiny"] = {"us_per_call": 1e3 * time_steps(fn, 200, stream), "host_us_per_call": host_us,
                       "device_us_per_call": dev_us, "launches": 1,
                       "note": "back-to-back calls, L2 warm; host_us includes the Python binding and "
                       "the C ABI's argument checks; device_us from a CUDA-graph replay of 20 calls"}
        del q, k, w, idx, sc, lg

    def _c4_fwd():
        wl = workloads.WORKLOADS["c4_fwd"]
        q, k, w = [t.cuda() for t in workloads.v4_inputs(wl, 0)]
        idx = torch.empty(wl.B, wl.S, wl.topk, dtype=torch.int32, device="cuda")
        sc = torch.empty_like(idx, dtype=torch.float32)
        lg = torch.empty(wl.B, wl.S, wl.Skv, dtype=torch.float32, device="cuda")
        fn = lambda: lidx.lidx_indexer_fwd(q, k, w, wl.ratio, wl.topk, materialise_logits=True,
                                           out=(idx, sc, lg))
        for _ in range(3):
            fn()
        ms = _median_ms(fn, stream, 10, flush)
        pairs = visible_pairs(wl.S, wl.Skv, wl.ratio, wl.B)
        fl = pairs * 2.0 * wl.H * wl.D
        alg_bytes = q.numel() * 2 + k.numel() * 2 + w.numel() * 4 + lg.numel() * 4 + idx.numel() * 8
        out["c4_fwd"] = {"ms": ms, "tflops": fl / ms / 1e9, "rows_per_s": wl.B * wl.S / ms * 1e3,
                         "tensor_frac": fl / ms / 1e9 / pk["bf16_tflops"],
                         "hbm_gbs": alg_bytes / ms / 1e6, "hbm_frac": alg_bytes / ms / 1e6 / pk["hbm_gbs"],
                         "l2": "256 MB flush before each launch"}
        # the same layer with the previous selection given (no selection; scores of those keys)
        given = idx.clone()
        ws = torch.empty(lidx.lidx_workspace_bytes(lidx.OP_INDEXER_FWD, wl.B, wl.S, wl.Skv, wl.H, wl.D,
                                                   wl.topk), dtype=torch.uint8, device="cuda")
        fn = lambda: lidx.lidx_indexer_fwd(q, k, w, wl.ratio, wl.topk, topk_indices=given,
                                           out=(idx, sc, None), workspace=ws)
        for _ in range(3):
            fn()
        ms = _median_ms(fn, stream, 10, flush)
        out["c4_fwd_given_indices"] = {"ms": ms, "tflops": fl / ms / 1e9,
                                       "tensor_frac": fl / ms / 1e9 / pk["bf16_tflops"],
                                       "note": "topk_indices given: same tensor-core sweep, the "
                                       "selection replaced by a gather", "l2": "256 MB flush"}
        del q, k, w, idx, sc, lg, given, ws

    def _v41_packed():
        # V4.1 packed documents: HBM-bound (q, allowed read; bf16 scores written)
        wl = workloads.WORKLOADS["v41_packed"]
        q, k, w, allowed = [t.cuda() for t in workloads.v41_inputs(wl, 0)]
        out16 = torch.empty(wl.B, wl.S, wl.Skv, dtype=torch.bfloat16, device="cuda")
        wsb = lidx.lidx_workspace_bytes(lidx.OP_SCORES_V41, wl.B, wl.S, wl.Skv, wl.H, wl.D)
        ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
        fn = lambda: lidx.lidx_indexer_scores_v41(q, k, w, allowed, out=out16, workspace=ws)
        for _ in range(3):
            fn()
        ms = _median_ms(fn, stream, 10, flush)
        vis = int(allowed.sum().item())
        alg_bytes = (q.numel() * 2 + k.numel() * 2 + w.numel() * 2 + allowed.numel() + out16.numel() * 2)
        out["v41_packed"] = {"ms": ms, "hbm_gbs": alg_bytes / ms / 1e6,
                             "hbm_frac": alg_bytes / ms / 1e6 / pk["hbm_gbs"],
                             "algorithmic_bytes": alg_bytes, "visible_pairs": vis,
                             "visible_pair_tflops": vis * 2.0 * wl.H * wl.D / ms / 1e9,
                             "launches": 1, "l2": "256 MB flush before each call"}
        tidx = torch.empty(wl.B, wl.S, wl.topk, dtype=torch.int32, device="cuda")
        tsc = torch.empty(wl.B, wl.S, wl.topk, dtype=torch.bfloat16, device="cuda")
        wsb = lidx.lidx_workspace_bytes(lidx.OP_TOPK_V41, wl.B, wl.S, wl.Skv, wl.H, wl.D, wl.topk, True)
        ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
        fn = lambda: lidx.lidx_indexer_topk_v41(q, k, w, allowed, wl.topk, out=(out16, tidx, tsc),
                                                workspace=ws)
        for _ in range(3):
            fn()
        ms2 = _median_ms(fn, stream, 10, flush)
        out["v41_packed_topk"] = {"ms": ms2, "topk": wl.topk, "selection_ms": ms2 - ms,
                                  "rows_per_s": wl.B * wl.S / ms2 * 1e3, "launches": 2,
                                  "l2": "256 MB flush before each call"}
        del q, k, w, allowed, out16, ws, tidx, tsc

    def _selection():
        # selection alone on adversarial rows: time of a tie-heavy row against a normal one
        rows, Skv, topk = 4096, 4096, 2048
        sel = {}
        for kind in ("normal", "ties", "const", "zero_pad", "two_values"):
            x = selection_rows(kind, rows, Skv).cuda()
            oi = torch.empty(rows, topk, dtype=torch.int32, device="cuda")
            os_ = torch.empty(rows, topk, dtype=torch.float32, device="cuda")
            fn = lambda: lidx.lidx_topk_rows(x, topk, out=(oi, os_))
            for _ in range(3):
                fn()
            sel[kind] = time_steps(fn, 10, stream)
            del x, oi, os_
        out["selection"] = {"rows": rows, "Skv": Skv, "topk": topk, "ms": sel,
                            "worst_over_normal": max(sel.values()) / sel["normal"],
                            "kernel": "topk_rows_kernel (standalone selection, 256 threads per row)"}

    def _bwd():
        # backward through the selected entries (selection: the forward's own top-k)
        wl = workloads.WORKLOADS["bwd"]
        q, k, w = [t.cuda() for t in workloads.v4_inputs(wl, 0)]
        idx, _, _ = lidx.lidx_indexer_fwd(q, k, w, wl.ratio, wl.topk)
        grad = workloads.grad_scores(wl.B, wl.S, wl.topk, 0).cuda()
        outs = (torch.empty(wl.S, wl.B, wl.H, wl.D, device="cuda"), torch.empty(wl.Skv, wl.B, wl.D, device="cuda"),
                torch.empty(wl.S, wl.B, wl.H, device="cuda"))
        wsb = lidx.lidx_workspace_bytes(lidx.OP_INDEXER_BWD, wl.B, wl.S, wl.Skv, wl.H, wl.D, wl.topk)
        ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
        fn = lambda: lidx.lidx_indexer_bwd(q, k, w, idx, grad, wl.ratio, out=outs, workspace=ws)
        for _ in range(2):
            fn()
        ms = time_steps(fn, 10, stream)
        nsel = int((idx >= 0).sum().item())
        fl = nsel * 6.0 * wl.H * wl.D
        out["bwd"] = {"ms": ms, "selected_pairs": nsel, "tflops": fl / ms / 1e9,
                      "tensor_frac": fl / ms / 1e9 / pk["bf16_tflops"], "kernel": BWD_KERNEL,
                      "launches": 4, "algorithmic": "6*H*D FLOP per selected pair",
                      "workspace_bytes": wsb}
        del q, k, w, idx, grad, outs, ws

    for name, f in (("tiny", _tiny), ("c4_fwd", _c4_fwd), ("v41_packed", _v41_packed),
                    ("selection", _selection), ("bwd", _bwd)):
        if names is None or name in names:
            f()
    return out

BWD_KERNEL = ("bwd_scatter_kernel + bwd_tile_kernel<64,0> (dq, dw) + bwd_tile_kernel<64,1> (dk partials) "
              "+ bwd_reduce_kernel; tcgen05, P as bf16 hi+lo from TMEM")


def run_gpu(args, wl, world, rank, local):
    import sparse_attention_top_tcgen05_gb300 as lidx

    pk, pk_src = peaks()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    q, k, w = workloads.v4_inputs(wl, args.seed + rank)
    qd, kd, wd = q.to(dev), k.to(dev), w.to(dev)
    B, S, H, D, Skv, topk = wl.B, wl.S, wl.H, wl.D, wl.Skv, wl.topk
    idx = torch.empty(B, S, topk, dtype=torch.int32, device=dev)
    sc = torch.empty(B, S, topk, dtype=torch.float32, device=dev)
    ws_bytes = lidx.lidx_workspace_bytes(lidx.OP_INDEXER_FWD, B, S, Skv, H, D, topk, False)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step_on(qb, kb, wb, ib, sb):
        lidx.lidx_indexer_fwd(qb, kb, wb, wl.ratio, topk, out=(ib, sb, None), workspace=ws)

    def step():
        step_on(qd, kd, wd, idx, sc)

    pairs = visible_pairs(S, Skv, wl.ratio, B)
    flops = pairs * 2.0 * H * D
    launches_per_step = 1

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert lidx.lidx_device_status() == 0
    barrier(world)
    with Clocks(local) as clk:
        torch.cuda.synchronize()
        ms = time_steps(step, args.steps, stream)
        torch.cuda.synchronize()
    barrier(world)
    status = lidx.lidx_device_status()
    ms_max = max_over_ranks(ms, world)
    value = world * flops / (ms_max * 1e-3) / 1e12
    rows_per_s = world * B * S / (ms_max * 1e-3)

    if args.no_e2e:
        e2e_ms = float("nan")
    else:
        e2e_ms = e2e_measure(q, k, w, (qd, kd, wd, idx, sc), step_on, args, world, stream)
    h2d = q.numel() * 2 + k.numel() * 2 + w.numel() * 4
    d2h = idx.numel() * 4 + sc.numel() * 4

    if rank != 0:
        return
    emit(args, wl, world, ms, ms_max, flops, pairs, value, rows_per_s, e2e_ms, h2d, d2h,
         launches_per_step, clk, status, pk, pk_src, lidx)


def e2e_measure(q, k, w, bufs, step_on, args, world, stream):
    """Same step through the C ABI with host buffers.

    Every step copies its inputs from pinned host memory and reads its top-k back into
    pinned host memory.  Consecutive steps overlap on three streams (host-to-device copy,
    compute, device-to-host copy) with two sets of device buffers, as a caller streaming
    batches would run them: step i's kernel starts only after its own inputs have landed,
    and step i+2 overwrites a buffer set only after step i's results were read back.
    """
    qh, kh, wh = q.pin_memory(), k.pin_memory(), w.pin_memory()
    sets = [bufs, tuple(torch.empty_like(t) for t in bufs)]
    outs_h = [(torch.empty(bufs[3].shape, dtype=torch.int32).pin_memory(),
               torch.empty(bufs[4].shape, dtype=torch.float32).pin_memory()) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    count = [0]

    def e2e_step():
        sl = count[0] & 1
        count[0] += 1
        qb, kb, wb, ib, sb = sets[sl]
        ih, sh = outs_h[sl]
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_comp[sl])  # step i-2 has finished reading this set
            qb.copy_(qh, non_blocking=True)
            kb.copy_(kh, non_blocking=True)
            wb.copy_(wh, non_blocking=True)
            ev_in[sl].record(s_in)
        with torch.cuda.stream(stream):
            stream.wait_event(ev_in[sl])
            stream.wait_event(ev_out[sl])  # step i-2's results have been read back
            step_on(qb, kb, wb, ib, sb)
            ev_comp[sl].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[sl])
            ih.copy_(ib, non_blocking=True)
            sh.copy_(sb, non_blocking=True)
            ev_out[sl].record(s_out)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 50))
    barrier(world)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    stream.wait_stream(s_out)
    end.record(stream)
    end.synchronize()
    ms = start.elapsed_time(end) / e2e_steps
    # the host copies must hold what the device path computed
    last = (count[0] - 1) & 1
    assert torch.equal(outs_h[last][0], bufs[3].cpu()) and torch.equal(
        outs_h[last][1].view(torch.int32), bufs[4].cpu().view(torch.int32)), "e2e outputs differ"
    return max_over_ranks(ms, world)


def emit(args, wl, world, ms, ms_max, flops, pairs, value, rows_per_s, e2e_ms, h2d, d2h,
         launches_per_step, clk, status, pk, pk_src, lidx):
    achieved = flops / (ms * 1e-3) / 1e12
    peak = pk["bf16_tflops"]
    traffic = recorded_traffic("score_fwd_kernel<64>/long_fused", SCORE_SRC)
    clocks = clk.summary()
    # the tensor pipe's nominal dense bf16 rate at the SM clock sampled during
    # the timed region: one 128x256x16 MMA (2^20 FLOP) per 128 cycles per SM
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    mhz = clocks.get("sm_mhz")
    at_clock = None
    if mhz:
        pipe = 8192.0 * sms * mhz * 1e6 / 1e12
        at_clock = {"peak": pipe, "frac": achieved / pipe, "unit": "TFLOP/s",
                    "basis": f"8192 FLOP/clk/SM x {sms} SMs x {mhz:.0f} MHz (median sampled)"}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_of(wl, world),
        "query_rows_per_s": rows_per_s, "valid_pairs_per_step": pairs * world,
        "tensor_peak_frac": achieved / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "score_fwd_kernel<64> (fused scoring + top-k)",
                     "peak_source": f"{pk_src} bf16_tflops (burst)",
                     "algorithmic": f"{pairs} visible pairs x 2*H*D = {flops:.4e} FLOP per launch",
                     "pipe_at_clock": at_clock},
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipeline": "copy in / compute / copy out on three streams, two device buffer sets"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "device_status": status,
    }
    if not args.no_side:
        line["other_workloads"] = side_workloads(lidx, pk, args.side.split(",") if args.side else None)
    if not args.no_cpu:
        line["cpu_baseline"] = cpu_oracle_sample(wl, args.cpu_stride)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_fused")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-stride", type=int, default=4)
    ap.add_argument("--B", type=int, default=0, help="override the workload's batch (profiling)")
    ap.add_argument("--S", type=int, default=0, help="override the workload's query length "
                    "(profiling); Skv follows as S // compress_ratio")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-side", action="store_true")
    ap.add_argument("--side", default="", help="comma-separated subset of the side measurements "
                    "(tiny, c4_fwd, v41_packed, selection, bwd); default all")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup()
    wl = workloads.WORKLOADS[args.workload]
    if args.B:
        wl = wl.with_(B=args.B)
    if args.S:
        wl = wl.with_(S=args.S, Skv=args.S // wl.ratio)
    if args.impl == "reference":
        run_reference(args, wl, world, rank)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA device (no CPU fallback)")
        run_gpu(args, wl, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
