"""Python binding of liblidx.so, the GB300 lightning-indexer library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI (``include/lidx.h``).  PyTorch supplies device
memory and the current stream.  There is no CPU fallback: if the library has
not been built, or no sm_103 device is present, calls raise.

Functions carry the C names:

  lidx_indexer_fwd          V4 forward: causal mask + per-row top-k
  lidx_indexer_fwd_ranges   V4 forward over explicit per-row [ks, ke) ranges
  lidx_indexer_logits       V4 logits only, causal or explicit [ks, ke) ranges
  lidx_extract_topk_scores  gather of logits at indices
  lidx_topk_rows            per-row top-k of given logits
  lidx_indexer_scores_v41   V4.1 bf16-rounded scores under a visibility mask
  lidx_indexer_topk_v41     V4.1 scores and their per-row top-k
  lidx_indexer_bwd          backward through the selected entries
  lidx_indexer_bwd_ranges   the same over explicit per-row ranges
  lidx_indexer_fwd_noalloc  fused forward with the library's own scratch
  lidx_workspace_bytes, lidx_device_status, lidx_status_string,
  lidx_set_wait_limit_ns, lidx_debug_stall_producer
"""

from __future__ import annotations

import ctypes as C
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblidx.so")

LIDX_OK = 0
STATUS = {0: "LIDX_OK", 1: "LIDX_ERR_NULL", 2: "LIDX_ERR_SHAPE", 3: "LIDX_ERR_ALIGN",
          4: "LIDX_ERR_UNSUPPORTED", 5: "LIDX_ERR_WORKSPACE", 6: "LIDX_ERR_CUDA",
          7: "LIDX_ERR_DEVICE_TIMEOUT", 8: "LIDX_ERR_NO_DEVICE"}
OP_INDEXER_FWD, OP_INDEXER_BWD, OP_SCORES_V41, OP_TOPK_V41 = 0, 1, 2, 3
ACT = {"relu": 0, "identity": 1}

# every symbol include/lidx.h declares
EXPORTS = ("lidx_indexer_fwd", "lidx_indexer_fwd_ranges", "lidx_indexer_logits",
           "lidx_extract_topk_scores", "lidx_topk_rows", "lidx_indexer_scores_v41",
           "lidx_indexer_topk_v41", "lidx_indexer_bwd", "lidx_indexer_bwd_ranges",
           "lidx_workspace_bytes", "lidx_device_status", "lidx_status_string", "lidx_version",
           "lidx_indexer_fwd_noalloc", "lidx_noalloc_scratch_bytes", "lidx_set_wait_limit_ns",
           "lidx_debug_stall_producer")


class LidxError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        msg = lib().lidx_status_string(status).decode() if _lib is not None else ""
        super().__init__(f"{call} returned {STATUS.get(status, status)}: {msg}")


_lib = None
_lock = threading.Lock()


def lib() -> C.CDLL:
    """The loaded library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m sparse_attention_top_tcgen05_gb300.build`")
            L = C.CDLL(LIB_PATH)
            P, i64, i32, sz = C.c_void_p, C.c_int64, C.c_int, C.c_size_t
            L.lidx_indexer_fwd.argtypes = [P, P, P, i64, i64, i64, i32, i32, i32, i32, i32,
                                           P, P, P, P, P, sz, P]
            L.lidx_indexer_fwd_ranges.argtypes = [P, P, P, i64, i64, i64, i32, i32, P, P, i32, i32,
                                                  P, P, P, P, P, sz, P]
            L.lidx_indexer_topk_v41.argtypes = [P, P, P, P, i64, i64, i64, i32, i32, i32, i32, P, P,
                                                P, P, sz, P]
            L.lidx_indexer_bwd_ranges.argtypes = [P, P, P, P, P, i64, i64, i64, i32, i32, P, P, i32,
                                                  i32, i32, P, P, P, P, sz, P]
            L.lidx_set_wait_limit_ns.argtypes = [C.c_uint64]
            L.lidx_set_wait_limit_ns.restype = C.c_uint64
            L.lidx_debug_stall_producer.argtypes = [i32]
            L.lidx_debug_stall_producer.restype = i32
            L.lidx_indexer_logits.argtypes = [P, P, P, i64, i64, i64, i32, i32, i32, P, P, i32,
                                              i32, P, P]
            L.lidx_extract_topk_scores.argtypes = [P, P, i64, i64, i64, i32, P, P]
            L.lidx_topk_rows.argtypes = [P, i64, i64, i64, i32, P, P, i32, P, P, P]
            L.lidx_indexer_scores_v41.argtypes = [P, P, P, P, i64, i64, i64, i32, i32, i32, P,
                                                  P, sz, P]
            L.lidx_indexer_bwd.argtypes = [P, P, P, P, P, i64, i64, i64, i32, i32, i32, i32, i32,
                                           i32, P, P, P, P, sz, P]
            L.lidx_indexer_fwd_noalloc.argtypes = [P, P, P, i64, i64, i64, i32, i32, i32, i32, i32,
                                                   P, P, P]
            L.lidx_indexer_fwd_noalloc.restype = i32
            L.lidx_noalloc_scratch_bytes.restype = sz
            L.lidx_workspace_bytes.argtypes = [i32, i64, i64, i64, i32, i32, i32, i32]
            L.lidx_workspace_bytes.restype = sz
            L.lidx_device_status.argtypes = [P]
            L.lidx_status_string.argtypes = [i32]
            L.lidx_status_string.restype = C.c_char_p
            L.lidx_version.restype = i32
            for name in ("lidx_indexer_fwd", "lidx_indexer_fwd_ranges", "lidx_indexer_logits",
                         "lidx_extract_topk_scores", "lidx_topk_rows", "lidx_indexer_scores_v41",
                         "lidx_indexer_topk_v41", "lidx_indexer_bwd", "lidx_indexer_bwd_ranges",
                         "lidx_device_status"):
                getattr(L, name).restype = i32
            _lib = L
    return _lib


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _need(t, name, dtype, dim):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check(rc, call):
    if rc != LIDX_OK:
        raise LidxError(rc, call)


def lidx_workspace_bytes(op, B, S, Skv, H, D, topk=0, logits_materialised=False) -> int:
    return int(lib().lidx_workspace_bytes(op, B, S, Skv, H, D, topk, int(bool(logits_materialised))))


def lidx_status_string(status: int) -> str:
    return lib().lidx_status_string(int(status)).decode()


def lidx_device_status(stream=None) -> int:
    return int(lib().lidx_device_status(_stream(stream)))


def _fwd_common(q, k, w, topk, topk_indices, materialise_logits, out, workspace):
    _need(q, "q", torch.bfloat16, 4)
    _need(k, "k", torch.bfloat16, 3)
    _need(w, "w", torch.float32, 3)
    S, B, H, D = q.shape
    Skv = k.shape[0]
    if k.shape[1] != B or k.shape[2] != D or tuple(w.shape) != (S, B, H):
        raise ValueError("q/k/w shapes disagree")
    if topk_indices is not None:
        _need(topk_indices, "topk_indices", torch.int32, 3)
    dev = q.device
    if out is None:
        idx = torch.empty(B, S, topk, dtype=torch.int32, device=dev)
        sc = torch.empty(B, S, topk, dtype=torch.float32, device=dev)
        lg = torch.empty(B, S, Skv, dtype=torch.float32, device=dev) if materialise_logits else None
    else:
        idx, sc, lg = out
    ws_bytes = lidx_workspace_bytes(OP_INDEXER_FWD, B, S, Skv, H, D, topk, lg is not None)
    if workspace is None and ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    return (S, B, H, D, Skv), idx, sc, lg, workspace, ws_bytes


def lidx_indexer_fwd(q, k, w, compress_ratio, topk, act="relu", topk_indices=None,
                     materialise_logits=False, stream=None, out=None, workspace=None):
    """V4 forward.  q [S,B,H,D] bf16, k [Skv,B,D] bf16, w [S,B,H] fp32.

    Returns (indices [B,S,topk] int32, scores [B,S,topk] fp32, logits or None).
    ``out`` may hold preallocated (indices, scores, logits) tensors.
    """
    (S, B, H, D, Skv), idx, sc, lg, workspace, ws_bytes = _fwd_common(
        q, k, w, topk, topk_indices, materialise_logits, out, workspace)
    rc = lib().lidx_indexer_fwd(_ptr(q), _ptr(k), _ptr(w), B, S, Skv, H, D, compress_ratio, topk,
                                ACT[act], _ptr(topk_indices), _ptr(lg), _ptr(idx), _ptr(sc),
                                _ptr(workspace), ws_bytes if workspace is not None else 0,
                                _stream(stream))
    _check(rc, "lidx_indexer_fwd")
    return idx, sc, lg


def lidx_indexer_fwd_ranges(q, k, w, ks, ke, topk, act="relu", topk_indices=None,
                            materialise_logits=False, stream=None, out=None, workspace=None):
    """V4 forward where row (b,s) sees keys [ks[s], ke[s]) (int32 [S] CUDA tensors)."""
    _need(ks, "ks", torch.int32, 1)
    _need(ke, "ke", torch.int32, 1)
    (S, B, H, D, Skv), idx, sc, lg, workspace, ws_bytes = _fwd_common(
        q, k, w, topk, topk_indices, materialise_logits, out, workspace)
    if ks.shape[0] != S or ke.shape[0] != S:
        raise ValueError("ks/ke must have S entries")
    rc = lib().lidx_indexer_fwd_ranges(_ptr(q), _ptr(k), _ptr(w), B, S, Skv, H, D, _ptr(ks), _ptr(ke),
                                       topk, ACT[act], _ptr(topk_indices), _ptr(lg), _ptr(idx),
                                       _ptr(sc), _ptr(workspace),
                                       ws_bytes if workspace is not None else 0, _stream(stream))
    _check(rc, "lidx_indexer_fwd_ranges")
    return idx, sc, lg


def lidx_indexer_fwd_noalloc(q, k, w, compress_ratio, topk, act="relu", stream=None, out=None):
    """The fused V4 forward using the library's own scratch array instead of a
    workspace, for callers that cannot allocate device memory.  Outputs may be
    passed in ``out`` = (indices, scores) so that the call allocates nothing."""
    _need(q, "q", torch.bfloat16, 4)
    _need(k, "k", torch.bfloat16, 3)
    _need(w, "w", torch.float32, 3)
    S, B, H, D = q.shape
    Skv = k.shape[0]
    if out is None:
        idx = torch.empty(B, S, topk, dtype=torch.int32, device=q.device)
        sc = torch.empty(B, S, topk, dtype=torch.float32, device=q.device)
    else:
        idx, sc = out
    rc = lib().lidx_indexer_fwd_noalloc(_ptr(q), _ptr(k), _ptr(w), B, S, Skv, H, D, compress_ratio,
                                        topk, ACT[act], _ptr(idx), _ptr(sc), _stream(stream))
    _check(rc, "lidx_indexer_fwd_noalloc")
    return idx, sc


def lidx_indexer_logits(q, k, w, compress_ratio=1, ks=None, ke=None, clean=True, act="relu",
                        stream=None, out=None):
    """Logits [B,S,Skv] fp32 over causal ranges or explicit per-row [ks, ke)."""
    _need(q, "q", torch.bfloat16, 4)
    _need(k, "k", torch.bfloat16, 3)
    _need(w, "w", torch.float32, 3)
    S, B, H, D = q.shape
    Skv = k.shape[0]
    if ks is not None:
        _need(ks, "ks", torch.int32, 1)
        _need(ke, "ke", torch.int32, 1)
    lg = torch.empty(B, S, Skv, dtype=torch.float32, device=q.device) if out is None else out
    rc = lib().lidx_indexer_logits(_ptr(q), _ptr(k), _ptr(w), B, S, Skv, H, D, compress_ratio,
                                   _ptr(ks), _ptr(ke), int(bool(clean)), ACT[act], _ptr(lg),
                                   _stream(stream))
    _check(rc, "lidx_indexer_logits")
    return lg


def lidx_extract_topk_scores(logits, idx, stream=None):
    _need(logits, "logits", torch.float32, 3)
    _need(idx, "idx", torch.int32, 3)
    B, S, Skv = logits.shape
    topk = idx.shape[2]
    out = torch.empty(B, S, topk, dtype=torch.float32, device=logits.device)
    rc = lib().lidx_extract_topk_scores(_ptr(logits), _ptr(idx), B, S, Skv, topk, _ptr(out),
                                        _stream(stream))
    _check(rc, "lidx_extract_topk_scores")
    return out


def lidx_topk_rows(logits, topk, compress_ratio=1, ks=None, ke=None, stream=None, out=None):
    """Top-k of each row of logits [B,S,Skv] (or [rows, Skv] with S = rows).

    Visible range per query s: causal from compress_ratio, or [ks[s], ke[s]).
    Returns (indices [..., topk] int32, scores [..., topk] fp32).
    """
    if logits.dim() == 3:
        B, S, Skv = logits.shape
    else:
        _need(logits, "logits", torch.float32, 2)
        B, (S, Skv) = 1, logits.shape
    if logits.dtype != torch.float32 or not logits.is_cuda or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous CUDA float32 tensor")
    if ks is not None:
        _need(ks, "ks", torch.int32, 1)
        _need(ke, "ke", torch.int32, 1)
    shape = tuple(logits.shape[:-1]) + (topk,)
    if out is None:
        idx = torch.empty(shape, dtype=torch.int32, device=logits.device)
        sc = torch.empty(shape, dtype=torch.float32, device=logits.device)
    else:
        idx, sc = out
    rc = lib().lidx_topk_rows(_ptr(logits), B * S, S, Skv, compress_ratio, _ptr(ks), _ptr(ke), topk,
                              _ptr(idx), _ptr(sc), _stream(stream))
    _check(rc, "lidx_topk_rows")
    return idx, sc


def lidx_indexer_scores_v41(q, k, w, allowed, act="relu", stream=None, out=None, workspace=None):
    """V4.1 scores bf16 [B,S,Skv].  q [B,S,H,D], k [B,Skv,D], w [B,S,H] bf16,
    allowed [B,S,Skv] bool."""
    _need(q, "q", torch.bfloat16, 4)
    _need(k, "k", torch.bfloat16, 3)
    _need(w, "w", torch.bfloat16, 3)
    if allowed.dtype not in (torch.bool, torch.uint8):
        raise TypeError("allowed must be bool or uint8")
    if not (allowed.is_cuda and allowed.is_contiguous() and allowed.dim() == 3):
        raise ValueError("allowed must be a contiguous CUDA [B,S,Skv] tensor")
    B, S, H, D = q.shape
    Skv = k.shape[1]
    res = torch.empty(B, S, Skv, dtype=torch.bfloat16, device=q.device) if out is None else out
    ws_bytes = lidx_workspace_bytes(OP_SCORES_V41, B, S, Skv, H, D)
    if workspace is None and ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    rc = lib().lidx_indexer_scores_v41(_ptr(q), _ptr(k), _ptr(w), _ptr(allowed), B, S, Skv, H, D,
                                       ACT[act], _ptr(res), _ptr(workspace),
                                       ws_bytes if workspace is not None else 0, _stream(stream))
    _check(rc, "lidx_indexer_scores_v41")
    return res


def lidx_indexer_topk_v41(q, k, w, allowed, topk, act="relu", keep_scores=True, stream=None,
                          out=None, workspace=None):
    """V4.1 scores and their per-row top-k.  Returns (scores bf16 [B,S,Skv] or
    None, indices int32 [B,S,topk], top-k scores bf16 [B,S,topk])."""
    _need(q, "q", torch.bfloat16, 4)
    _need(k, "k", torch.bfloat16, 3)
    _need(w, "w", torch.bfloat16, 3)
    if allowed.dtype not in (torch.bool, torch.uint8):
        raise TypeError("allowed must be bool or uint8")
    if not (allowed.is_cuda and allowed.is_contiguous() and allowed.dim() == 3):
        raise ValueError("allowed must be a contiguous CUDA [B,S,Skv] tensor")
    B, S, H, D = q.shape
    Skv = k.shape[1]
    dev = q.device
    if out is None:
        res = torch.empty(B, S, Skv, dtype=torch.bfloat16, device=dev) if keep_scores else None
        idx = torch.empty(B, S, topk, dtype=torch.int32, device=dev)
        tsc = torch.empty(B, S, topk, dtype=torch.bfloat16, device=dev)
    else:
        res, idx, tsc = out
    ws_bytes = lidx_workspace_bytes(OP_TOPK_V41, B, S, Skv, H, D, topk, res is not None)
    if workspace is None and ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    rc = lib().lidx_indexer_topk_v41(_ptr(q), _ptr(k), _ptr(w), _ptr(allowed), B, S, Skv, H, D,
                                     ACT[act], topk, _ptr(res), _ptr(idx), _ptr(tsc), _ptr(workspace),
                                     ws_bytes if workspace is not None else 0, _stream(stream))
    _check(rc, "lidx_indexer_topk_v41")
    return res, idx, tsc


def lidx_set_wait_limit_ns(ns: int) -> int:
    """Limit of every in-kernel pipeline wait (0: the 2 s default); returns the previous."""
    return int(lib().lidx_set_wait_limit_ns(int(ns)))


def lidx_debug_stall_producer(on: bool) -> int:
    """Test switch: the scoring kernel's producer loads nothing, so its waits run out."""
    return int(lib().lidx_debug_stall_producer(int(bool(on))))


def _bwd_common(q, k, w, idx, grad, grad_dtype, out, workspace):
    _need(q, "q", torch.bfloat16, 4)
    _need(k, "k", torch.bfloat16, 3)
    _need(w, "w", torch.float32, 3)
    _need(idx, "idx", torch.int32, 3)
    _need(grad, "grad", torch.float32, 3)
    S, B, H, D = q.shape
    Skv = k.shape[0]
    topk = idx.shape[2]
    dev = q.device
    gdt = {torch.float32: 0, torch.bfloat16: 1}[grad_dtype]
    if out is None:
        dq = torch.empty(S, B, H, D, dtype=grad_dtype, device=dev)
        dk = torch.empty(Skv, B, D, dtype=grad_dtype, device=dev)
        dw = torch.empty(S, B, H, dtype=torch.float32, device=dev)
    else:
        dq, dk, dw = out
    ws_bytes = lidx_workspace_bytes(OP_INDEXER_BWD, B, S, Skv, H, D, topk)
    if workspace is None and ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    return (S, B, H, D, Skv, topk, gdt), dq, dk, dw, workspace, ws_bytes


def lidx_indexer_bwd_ranges(q, k, w, idx, grad, ks, ke, act="relu", grad_dtype=torch.float32,
                            stream=None, out=None, workspace=None):
    """Backward where row (b,s) sees keys [ks[s], ke[s]); dk is this call's partial sum."""
    _need(ks, "ks", torch.int32, 1)
    _need(ke, "ke", torch.int32, 1)
    (S, B, H, D, Skv, topk, gdt), dq, dk, dw, workspace, ws_bytes = _bwd_common(
        q, k, w, idx, grad, grad_dtype, out, workspace)
    rc = lib().lidx_indexer_bwd_ranges(_ptr(q), _ptr(k), _ptr(w), _ptr(idx), _ptr(grad), B, S, Skv, H,
                                       D, _ptr(ks), _ptr(ke), topk, ACT[act], gdt, _ptr(dq), _ptr(dk),
                                       _ptr(dw), _ptr(workspace),
                                       ws_bytes if workspace is not None else 0, _stream(stream))
    _check(rc, "lidx_indexer_bwd_ranges")
    return dq, dk, dw


def lidx_indexer_bwd(q, k, w, idx, grad, compress_ratio, act="relu", grad_dtype=torch.float32,
                     stream=None, out=None, workspace=None):
    """Gradients (dq [S,B,H,D], dk [Skv,B,D] in grad_dtype (fp32 or bf16), dw [S,B,H] fp32)."""
    (S, B, H, D, Skv, topk, gdt), dq, dk, dw, workspace, ws_bytes = _bwd_common(
        q, k, w, idx, grad, grad_dtype, out, workspace)
    rc = lib().lidx_indexer_bwd(_ptr(q), _ptr(k), _ptr(w), _ptr(idx), _ptr(grad), B, S, Skv, H, D,
                                compress_ratio, topk, ACT[act], gdt, _ptr(dq), _ptr(dk), _ptr(dw),
                                _ptr(workspace), ws_bytes if workspace is not None else 0,
                                _stream(stream))
    _check(rc, "lidx_indexer_bwd")
    return dq, dk, dw
