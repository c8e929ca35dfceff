"""CPU checks of the C ABI: the library builds, loads, exports every symbol
include/lidx.h declares, and rejects bad arguments before touching a GPU."""

import ctypes as C
import os
import re

import pytest

import sparse_attention_top_tcgen05_gb300 as lidx
from sparse_attention_top_tcgen05_gb300 import build as lidx_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    lidx_build.build()
    return lidx.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "lidx.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lidx_[a-z0-9_]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert sorted(lidx.EXPORTS) == header_functions()


def test_library_exports_every_header_symbol(L):
    for name in header_functions():
        assert hasattr(L, name), name


def test_version_and_status_strings(L):
    assert L.lidx_version() == 0x000200
    for code in range(0, 9):
        s = lidx.lidx_status_string(code)
        assert s and s != "unknown status"
    assert lidx.lidx_status_string(99) == "unknown status"


def _fwd(L, **kw):
    a = dict(q=16, k=16, w=16, B=1, S=8, Skv=4, H=8, D=32, r=4, topk=2, act=0, tin=None,
             lg=None, idx=16, sc=16, ws=None, wsb=0)
    a.update(kw)
    P = lambda v: None if v is None else C.c_void_p(v)
    return L.lidx_indexer_fwd(P(a["q"]), P(a["k"]), P(a["w"]), a["B"], a["S"], a["Skv"], a["H"],
                              a["D"], a["r"], a["topk"], a["act"], P(a["tin"]), P(a["lg"]),
                              P(a["idx"]), P(a["sc"]), P(a["ws"]), a["wsb"], None)


def test_argument_validation_without_gpu(L):
    # rules are checked before any device query, so these run on a CPU host
    assert _fwd(L, q=None) == 1                       # NULL
    assert _fwd(L, H=6) == 2                          # heads not a power of two
    assert _fwd(L, H=256) == 2                        # heads > 128
    assert _fwd(L, D=24) == 2                         # index_dim % 16 != 0
    assert _fwd(L, D=0) == 2
    assert _fwd(L, topk=0) == 2
    assert _fwd(L, r=0) == 2
    assert _fwd(L, B=0) == 2
    assert _fwd(L, act=5) == 2
    assert _fwd(L, q=18) == 3                         # misaligned
    assert _fwd(L, Skv=70000) == 4                    # beyond this build's selection span
    assert _fwd(L, Skv=70000, tin=16) != 4            # no selection with given indices
    assert _fwd(L, B=1 << 16, S=1 << 16) == 2         # rows (b, s) must fit an int


def test_new_entry_points_validate_without_gpu(L):
    P = C.c_void_p
    # explicit ranges need both arrays
    rc = L.lidx_indexer_fwd_ranges(P(16), P(16), P(16), 1, 8, 4, 8, 32, None, P(16), 2, 0, None, None,
                                   P(16), P(16), None, 0, None)
    assert rc == 1
    # V4.1 top-k: topk 0 and a misaligned query pointer are rejected before any launch
    args = [P(16), P(16), P(16), P(16), 1, 8, 64, 8, 32, 0]
    assert L.lidx_indexer_topk_v41(*args, 0, None, P(16), P(16), None, 0, None) == 2
    args[0] = P(18)
    assert L.lidx_indexer_topk_v41(*args, 4, None, P(16), P(16), None, 0, None) == 3
    # backward ranges need both arrays; grad_dtype outside {0, 1} is a shape error
    rc = L.lidx_indexer_bwd_ranges(P(16), P(16), P(16), P(16), P(16), 1, 8, 4, 8, 32, P(16), None, 2,
                                   0, 0, P(16), P(16), P(16), None, 0, None)
    assert rc == 1
    rc = L.lidx_indexer_bwd(P(16), P(16), P(16), P(16), P(16), 1, 8, 4, 8, 32, 4, 2, 0, 7, P(16),
                            P(16), P(16), None, 0, None)
    assert rc == 2


def test_wait_limit_and_stall_switch_round_trip(L):
    old = lidx.lidx_set_wait_limit_ns(1000)
    assert old == 2_000_000_000
    assert lidx.lidx_set_wait_limit_ns(0) == 1000          # 0 restores the default
    assert lidx.lidx_set_wait_limit_ns(0) == 2_000_000_000
    assert lidx.lidx_debug_stall_producer(True) == 0
    assert lidx.lidx_debug_stall_producer(False) == 1


def test_workspace_sizes(L):
    assert lidx.lidx_workspace_bytes(lidx.OP_INDEXER_FWD, 2, 16384, 4096, 64, 128, 2048, True) == 0
    ws = lidx.lidx_workspace_bytes(lidx.OP_INDEXER_FWD, 2, 16384, 4096, 64, 128, 2048, False)
    assert ws >= 148 * 4 * 4096 * 4  # one 4-row x Skv fp32 buffer per CTA at least


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(lidx, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(lidx, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        lidx.lib()
