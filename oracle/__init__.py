"""ctypes front end of the plain C CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The CUDA library never imports this.

Inputs are CPU torch tensors or numpy arrays; bf16 tensors are passed as their
raw 16-bit patterns.  Outputs are numpy arrays (fp64 unless stated).
"""

from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liblidx_oracle.so")
_lib = None
_lock = threading.Lock()

ACT = {"relu": 0, "identity": 1}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/_build (no vendor code involved)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    hdr = os.path.join(_HERE, "oracle.h")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC), os.path.getmtime(hdr))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            P = C.c_void_p
            i64, i32, dbl = C.c_int64, C.c_int, C.c_double
            L.orc_set_threads.argtypes = [i32]
            L.orc_get_threads.restype = i32
            L.orc_bf16_round.argtypes = [dbl]
            L.orc_bf16_round.restype = dbl
            L.orc_bf16_round_array.argtypes = [P, P, i64]
            L.orc_causal_ranges.argtypes = [i64, i64, i32, P, P]
            L.orc_logits_rows.argtypes = [P, P, P, i64, i64, i64, i32, i32, P, P, i32, P, i64, P]
            L.orc_topk_rows.argtypes = [P, i64, i64, P, i64, P, P, i32, P, P]
            L.orc_extract_rows.argtypes = [P, i64, i64, P, i32, P]
            L.orc_topk_masked_rows.argtypes = [P, P, i64, i64, i32, P, P]
            L.orc_gather_scores_rows.argtypes = [P, P, P, i64, i64, i64, i32, i32, P, P, i32,
                                                 P, i64, P, i32, P]
            L.orc_scores_v41_rows.argtypes = [P, P, P, P, i64, i64, i64, i32, i32, i32, P, i64, P]
            L.orc_bwd.argtypes = [P, P, P, P, P, i64, i64, i64, i32, i32, P, P, i32, i32, dbl,
                                  P, P, P, P, P, P]
            _lib = L
    return _lib


def _np(x, dtype):
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu()
        if x.dtype == torch.bfloat16:
            x = x.view(torch.int16)
        x = x.numpy()
    return np.ascontiguousarray(x, dtype=dtype)


def _p(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def get_threads() -> int:
    return int(lib().orc_get_threads())


def bf16_round(x) -> np.ndarray:
    a = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(a)
    lib().orc_bf16_round_array(_p(a), _p(out), a.size)
    return out


def causal_ranges(S: int, Skv: int, ratio: int):
    ks = np.empty(S, np.int32)
    ke = np.empty(S, np.int32)
    lib().orc_causal_ranges(S, Skv, ratio, _p(ks), _p(ke))
    return ks, ke


def _rows(rows, B, S):
    if rows is None:
        return np.arange(B * S, dtype=np.int64)
    return np.ascontiguousarray(rows, dtype=np.int64)


def logits_rows(q, k, w, ks, ke, act="relu", rows=None):
    """fp64 masked logits for rows r=b*S+s of SBHD q [S,B,H,D], k [Skv,B,D], w [S,B,H]."""
    S, B, H, D = q.shape
    Skv = k.shape[0]
    qa, ka, wa = _np(q, np.uint16), _np(k, np.uint16), _np(w, np.float32)
    ksa, kea = _np(ks, np.int32), _np(ke, np.int32)
    r = _rows(rows, B, S)
    out = np.empty((r.size, Skv), np.float64)
    rc = lib().orc_logits_rows(_p(qa), _p(ka), _p(wa), B, S, Skv, H, D, _p(ksa), _p(kea),
                               ACT[act], _p(r), r.size, _p(out))
    assert rc == 0
    return out


def topk_rows(logits, S, ks, ke, topk, rows):
    """Top-k of each row of ``logits`` [nrows, Skv] over its visible range."""
    lg = _np(logits, np.float64)
    nrows, Skv = lg.shape
    r = _np(rows, np.int64)
    ksa, kea = _np(ks, np.int32), _np(ke, np.int32)
    idx = np.empty((nrows, topk), np.int32)
    sc = np.empty((nrows, topk), np.float64)
    rc = lib().orc_topk_rows(_p(lg), nrows, Skv, _p(r), S, _p(ksa), _p(kea), topk, _p(idx), _p(sc))
    assert rc == 0
    return idx, sc


def topk_masked_rows(logits, mask, topk):
    """Top-k of each row of ``logits`` [nrows, Skv] over the entries where
    ``mask`` [nrows, Skv] is nonzero; padding -1 / -inf."""
    lg = _np(logits, np.float64)
    nrows, Skv = lg.shape
    m = _np(mask, np.uint8).reshape(nrows, Skv)
    idx = np.empty((nrows, topk), np.int32)
    sc = np.empty((nrows, topk), np.float64)
    rc = lib().orc_topk_masked_rows(_p(lg), _p(m), nrows, Skv, topk, _p(idx), _p(sc))
    assert rc == 0
    return idx, sc


def extract_rows(logits, idx):
    lg = _np(logits, np.float64)
    ia = _np(idx, np.int32)
    nrows, Skv = lg.shape
    topk = ia.shape[-1]
    out = np.empty((nrows, topk), np.float64)
    lib().orc_extract_rows(_p(lg), nrows, Skv, _p(ia.reshape(nrows, topk)), topk, _p(out))
    return out


def gather_scores_rows(q, k, w, ks, ke, idx, act="relu", rows=None):
    S, B, H, D = q.shape
    Skv = k.shape[0]
    qa, ka, wa = _np(q, np.uint16), _np(k, np.uint16), _np(w, np.float32)
    ksa, kea = _np(ks, np.int32), _np(ke, np.int32)
    r = _rows(rows, B, S)
    ia = _np(idx, np.int32).reshape(r.size, -1)
    topk = ia.shape[1]
    out = np.empty((r.size, topk), np.float64)
    rc = lib().orc_gather_scores_rows(_p(qa), _p(ka), _p(wa), B, S, Skv, H, D, _p(ksa), _p(kea),
                                      ACT[act], _p(r), r.size, _p(ia), topk, _p(out))
    assert rc == 0
    return out


def indexer_fwd_rows(q, k, w, ratio, topk, act="relu", rows=None):
    """V4 forward (causal ranges, logits, top-k) for the given rows.

    Returns (idx [n,topk] int32, scores [n,topk] fp64, logits [n,Skv] fp64).
    """
    S, B = q.shape[0], q.shape[1]
    Skv = k.shape[0]
    ks, ke = causal_ranges(S, Skv, ratio)
    r = _rows(rows, B, S)
    lg = logits_rows(q, k, w, ks, ke, act, r)
    idx, sc = topk_rows(lg, S, ks, ke, topk, r)
    return idx, sc, lg


def scores_v41_rows(q, k, w, allowed, act="relu", rows=None):
    """V4.1 bf16 scores (as float32) for rows of BSHD q [B,S,H,D]."""
    B, S, H, D = q.shape
    Skv = k.shape[1]
    qa, ka, wa = _np(q, np.uint16), _np(k, np.uint16), _np(w, np.uint16)
    al = _np(allowed, np.uint8)
    r = _rows(rows, B, S)
    out = np.empty((r.size, Skv), np.float32)
    rc = lib().orc_scores_v41_rows(_p(qa), _p(ka), _p(wa), _p(al), B, S, Skv, H, D, ACT[act],
                                   _p(r), r.size, _p(out))
    assert rc == 0
    return out


def bwd(q, k, w, idx, grad, ks, ke, act="relu", gamma=None, slack=True):
    """Gradients (dq [S,B,H,D], dk [Skv,B,D], dw [S,B,H]) in fp64, plus the
    per-element slack for ReLU decisions within float32 accumulation error."""
    S, B, H, D = q.shape
    Skv = k.shape[0]
    topk = idx.shape[-1]
    if gamma is None:
        gamma = D * 2.0 ** -22
    qa, ka, wa = _np(q, np.uint16), _np(k, np.uint16), _np(w, np.float32)
    ia, ga = _np(idx, np.int32), _np(grad, np.float32)
    ksa, kea = _np(ks, np.int32), _np(ke, np.int32)
    dq = np.empty((S, B, H, D)); dk = np.empty((Skv, B, D)); dw = np.empty((S, B, H))
    if slack:
        sq, sk, sw = np.empty_like(dq), np.empty_like(dk), np.empty_like(dw)
        ptrs = (_p(sq), _p(sk), _p(sw))
    else:
        sq = sk = sw = None
        ptrs = (None, None, None)
    rc = lib().orc_bwd(_p(qa), _p(ka), _p(wa), _p(ia), _p(ga), B, S, Skv, H, D, _p(ksa), _p(kea),
                       topk, ACT[act], float(gamma), _p(dq), _p(dk), _p(dw), *ptrs)
    assert rc == 0
    return dq, dk, dw, sq, sk, sw
