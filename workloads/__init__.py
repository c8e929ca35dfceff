"""Seeded synthetic inputs for the lightning-indexer hot path.

This module only draws random numbers and lays them out in the layouts the
indexer pages give (SBHD queries, [seqlen_kv, batch, dim] keys, ...).  It holds
none of the method's arithmetic: no dot products, no activation, no masking
rule, no top-k.  Both the CPU oracle (``oracle/``) and the CUDA path consume the
tensors built here, so it is the only code the two sides share.

Distributions follow the five workloads the indexer is measured on:

* ``tiny``       B=1 S=256  H=8  D=32  ratio 4, Skv=64,   topk=16,  q,k ~ N(0,1)
* ``c4_fwd``     B=1 S=4096 H=64 D=128 ratio 4, Skv=1024, topk=512, q,k ~ N(0,1/D)
* ``long_fused`` B=2 S=16384 H=64 D=128 ratio 4, Skv=4096, topk=2048
* ``v41_packed`` B=1 S=8192 Skv=8192 H=64 D=128, packed documents, query offset 24576;
  the selection on its scores keeps topk=512 per row
* ``bwd``        B=1 S=8192 H=64 D=128 ratio 4, Skv=2048, topk=1024

Weights are N(0,1)/sqrt(H).  Values are drawn in float32 and rounded to bf16
with round-to-nearest-even by torch's dtype conversion.  Streams: q=1, k=2,
w=3, grad=4, docs=5, selection=6, all keyed on (seed, stream).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch

STREAM_Q, STREAM_K, STREAM_W, STREAM_GRAD, STREAM_DOCS, STREAM_SEL = 1, 2, 3, 4, 5, 6


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    S: int
    H: int
    D: int
    Skv: int
    ratio: int = 4
    topk: int = 0
    qk_std: float = 1.0
    w_std: float = 1.0
    materialise_logits: bool = False
    # packed-document visibility (V4.1 only)
    query_offset: int = 0
    doc_min: int = 0
    doc_max: int = 0
    kind: str = "v4"  # "v4" | "v41" | "bwd"
    extra: dict = field(default_factory=dict)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def _w(name, **kw):
    return Workload(name=name, **kw)


WORKLOADS = {
    "tiny": _w("tiny", B=1, S=256, H=8, D=32, Skv=64, ratio=4, topk=16,
               qk_std=1.0, w_std=1.0 / math.sqrt(8), materialise_logits=True),
    "c4_fwd": _w("c4_fwd", B=1, S=4096, H=64, D=128, Skv=1024, ratio=4, topk=512,
                 qk_std=1.0 / math.sqrt(128), w_std=1.0 / 8, materialise_logits=True),
    "long_fused": _w("long_fused", B=2, S=16384, H=64, D=128, Skv=4096, ratio=4, topk=2048,
                     qk_std=1.0 / math.sqrt(128), w_std=1.0 / 8, materialise_logits=False),
    "v41_packed": _w("v41_packed", B=1, S=8192, H=64, D=128, Skv=8192, ratio=4, topk=512,
                     qk_std=1.0 / math.sqrt(128), w_std=1.0 / 8, query_offset=24576,
                     doc_min=512, doc_max=4096, kind="v41"),
    "bwd": _w("bwd", B=1, S=8192, H=64, D=128, Skv=2048, ratio=4, topk=1024,
              qk_std=1.0 / math.sqrt(128), w_std=1.0 / 8, kind="bwd"),
}


def rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(stream)])


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """float32 array -> bf16 tensor (round to nearest even, torch conversion)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def normal(seed, stream, shape, std) -> np.ndarray:
    return (rng(seed, stream).standard_normal(size=shape, dtype=np.float32) * np.float32(std))


def v4_inputs(wl: Workload, seed: int = 0):
    """q [S,B,H,D] bf16, k [Skv,B,D] bf16, w [S,B,H] fp32 (CPU tensors)."""
    q = to_bf16(normal(seed, STREAM_Q, (wl.S, wl.B, wl.H, wl.D), wl.qk_std))
    k = to_bf16(normal(seed, STREAM_K, (wl.Skv, wl.B, wl.D), wl.qk_std))
    w = torch.from_numpy(normal(seed, STREAM_W, (wl.S, wl.B, wl.H), wl.w_std))
    return q, k, w


def integer_inputs(B, S, Skv, H, D, seed=0, layout="sbhd"):
    """Integer-valued q,k in {-2..2} and w in {+-1/4, +-1/2, +-1}.

    With such values every product and every partial sum the scoring performs
    is exactly representable in float32, whatever the summation order, so a
    float32 implementation must reproduce the exact result bit for bit.
    """
    g = rng(seed, 11)
    qv = g.integers(-2, 3, size=(S, B, H, D)).astype(np.float32)
    kv = g.integers(-2, 3, size=(Skv, B, D)).astype(np.float32)
    wv = g.choice(np.array([-1.0, -0.5, -0.25, 0.25, 0.5, 1.0], np.float32), size=(S, B, H))
    if layout == "bshd":
        qv = np.ascontiguousarray(qv.transpose(1, 0, 2, 3))
        kv = np.ascontiguousarray(kv.transpose(1, 0, 2))
        wv = np.ascontiguousarray(wv.transpose(1, 0, 2))
    return to_bf16(qv), to_bf16(kv), torch.from_numpy(np.ascontiguousarray(wv))


def doc_starts(total_tokens: int, doc_min: int, doc_max: int, seed: int) -> np.ndarray:
    """Start token of the document each token belongs to.

    Documents are laid end to end over the global token stream with lengths
    drawn uniformly from [doc_min, doc_max]; the last one is cut at the end.
    """
    g = rng(seed, STREAM_DOCS)
    starts = np.empty(total_tokens, dtype=np.int64)
    pos = 0
    while pos < total_tokens:
        ln = int(g.integers(doc_min, doc_max + 1))
        end = min(total_tokens, pos + ln)
        starts[pos:end] = pos
        pos = end
    return starts


def v41_allowed(wl: Workload, seed: int = 0) -> torch.Tensor:
    """bool visibility [B,S,Skv] for packed documents under global causality.

    Query s sits at global token p = query_offset + s.  Compressed key t covers
    tokens [ratio*t, ratio*t + ratio).  Key t is visible to p when its group is
    complete before p (t < (p+1)//ratio) and starts inside p's document.
    This stands in for the attention-metadata path that builds the tensor.
    """
    total = wl.ratio * wl.Skv
    out = np.zeros((wl.B, wl.S, wl.Skv), dtype=np.bool_)
    t = np.arange(wl.Skv, dtype=np.int64)
    for b in range(wl.B):
        starts = doc_starts(total, wl.doc_min, wl.doc_max, seed + 1000 * b)
        p = wl.query_offset + np.arange(wl.S, dtype=np.int64)
        hi = np.minimum((p + 1) // wl.ratio, wl.Skv)
        lo = (starts[np.minimum(p, total - 1)] + wl.ratio - 1) // wl.ratio
        out[b] = (t[None, :] >= lo[:, None]) & (t[None, :] < hi[:, None])
    return torch.from_numpy(out)


def v41_inputs(wl: Workload, seed: int = 0):
    """q [B,S,H,D] bf16, k [B,Skv,D] bf16, w [B,S,H] bf16, allowed [B,S,Skv] bool."""
    q = to_bf16(normal(seed, STREAM_Q, (wl.B, wl.S, wl.H, wl.D), wl.qk_std))
    k = to_bf16(normal(seed, STREAM_K, (wl.B, wl.Skv, wl.D), wl.qk_std))
    w = to_bf16(normal(seed, STREAM_W, (wl.B, wl.S, wl.H), wl.w_std))
    return q, k, w, v41_allowed(wl, seed)


def random_selection(B: int, S: int, Skv: int, topk: int, counts, seed: int = 0):
    """Synthetic top-k selection [B,S,topk] int32.

    Row s draws min(topk, counts[s]) distinct keys from [0, counts[s]) in random
    order and pads the rest with -1.  ``counts`` (visible keys per row) comes
    from the caller, so this module stays free of the masking rule.  It stands
    in for a forward pass's selected indices when driving the backward.
    """
    g = rng(seed, STREAM_SEL)
    n = np.asarray(counts, dtype=np.int64).reshape(S)
    idx = np.full((B, S, topk), -1, dtype=np.int32)
    cols = np.arange(Skv)[None, :]
    for b in range(B):
        keys = g.random((S, Skv), dtype=np.float32)
        keys[cols >= n[:, None]] = 2.0  # keys past the row's count sort last
        order = np.argsort(keys, axis=1, kind="stable")[:, :topk].astype(np.int32)
        if order.shape[1] < topk:  # fewer keys than slots: pad the tail
            order = np.pad(order, ((0, 0), (0, topk - order.shape[1])), constant_values=-1)
        cnt = np.minimum(n, topk)
        valid = np.arange(topk)[None, :] < cnt[:, None]
        idx[b] = np.where(valid, order, -1)
    return torch.from_numpy(idx)


def grad_scores(B: int, S: int, topk: int, seed: int = 0) -> torch.Tensor:
    return torch.from_numpy(normal(seed, STREAM_GRAD, (B, S, topk), 1.0))


def bwd_inputs(wl: Workload, counts, seed: int = 0):
    """q, k, w as the forward, a synthetic selection of ``counts`` keys per row
    and grad_scores ~ N(0,1) [B,S,topk] fp32."""
    q, k, w = v4_inputs(wl, seed)
    idx = random_selection(wl.B, wl.S, wl.Skv, wl.topk, counts, seed)
    g = grad_scores(wl.B, wl.S, wl.topk, seed)
    return q, k, w, idx, g


def sample_rows(B: int, S: int, stride: int, offset: int = 0) -> np.ndarray:
    """Row ids b*S + s for every ``stride``-th query row of every batch, always
    including the last row of each batch (the longest causal range)."""
    rows = []
    for b in range(B):
        ss = list(range(offset, S, stride))
        if S - 1 not in ss:
            ss.append(S - 1)
        rows.extend(b * S + s for s in ss)
    return np.asarray(rows, dtype=np.int64)
