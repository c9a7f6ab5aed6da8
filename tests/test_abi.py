"""libfkl.so loads, exports every function include/fkl.h declares, and rejects bad
arguments on the host before touching a GPU.  No compute call is made here."""
import ctypes
import os
import re

import pytest

from lm_head_kl_fkl_b300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fkl.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fkl_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(_lib.LIB_PATH):
        from lm_head_kl_fkl_b300 import build
        build.build(quiet=True)
    return _lib.lib()


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert "fkl_forward" in names and "fkl_backward" in names
    for n in names:
        assert hasattr(L, n), f"{n} declared in fkl.h but not exported"
    assert set(names) == set(_lib.SIGNATURES), "binding signatures drift from the header"


def test_no_extra_exports(L):
    # the library exports exactly the C ABI under the fkl_ prefix (plus nothing C++ mangled-public)
    out = os.popen(f"nm -D --defined-only {_lib.LIB_PATH}").read()
    fkl_syms = sorted(set(re.findall(r"\bT (fkl_\w+)", out)))
    assert fkl_syms == declared_functions()


def test_status_strings(L):
    for code in range(7):
        assert L.fkl_status_string(code).decode()
    assert L.fkl_status_string(3).decode().startswith("teacher index")


def test_workspace_size_arithmetic(L):
    ws = L.fkl_workspace_size
    # bounded by the chunk, not by N (apart from 4 bytes per token)
    a = ws(32768, 2880, 201088, 100, 0)
    b = ws(131072, 2880, 201088, 100, 0)
    assert 0 < a <= b and b - a <= (131072 - 32768) * 4 + 4096
    # the memory-stress shape stays under 2 GB of workspace
    assert b < 2_000_000_000
    # a smaller chunk needs less
    assert ws(32768, 2880, 201088, 100, 1024) < a
    # invalid sizes give 0
    for args in [(0, 64, 100, 4, 0), (10, 60, 100, 4, 0), (10, 64, 100, 0, 0), (10, 64, 100, 300, 0),
                 (10, 64, 3, 4, 0), (10, 64, 100, 4, 100), (10, 64, 100, 4, -128)]:
        assert ws(*args) == 0, args


def _fwd(L, **kw):
    a = dict(h=16, W=16, idx=16, t=16, mask=None, N=10, d=64, V=100, K=4, T=1.0, chunk=0,
             loss=16, lse=16, ws=16, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    c = ctypes.c_void_p
    return L.fkl_forward(c(a["h"]), c(a["W"]), c(a["idx"]), c(a["t"]), c(a["mask"]), a["N"], a["d"],
                         a["V"], a["K"], a["T"], a["chunk"], c(a["loss"]), c(a["lse"]), c(a["ws"]),
                         a["ws_bytes"], c(a["stream"]))


@pytest.mark.parametrize("kw", [
    dict(h=None), dict(W=None), dict(idx=None), dict(t=None), dict(ws=None), dict(loss=None),
    dict(lse=None), dict(N=0), dict(d=12), dict(K=0), dict(K=257), dict(V=3), dict(T=0.0),
    dict(T=float("nan")), dict(T=-1.0), dict(chunk=100), dict(h=24), dict(ws=8),
])
def test_forward_rejects_invalid_arguments(L, kw):
    assert _fwd(L, **kw) == 1  # FKL_ERR_INVALID_ARG, decided before any CUDA call
    assert L.fkl_last_error().decode()


def test_forward_rejects_small_workspace(L):
    assert _fwd(L, ws_bytes=1000) == 2  # FKL_ERR_WORKSPACE
    assert b"needed" in L.fkl_last_error()


def test_backward_rejects_invalid_arguments(L):
    c = ctypes.c_void_p
    st = L.fkl_backward(c(16), c(16), c(16), c(16), None, 10, 64, 100, 4, 1.0, 0, c(16), None,
                        None, c(16), c(16), 1 << 30, None)
    assert st == 1
    st = L.fkl_backward(c(16), c(16), c(16), c(16), None, 10, 64, 100, 4, 1.0, 0, c(16), None,
                        c(24), c(16), c(16), 1 << 30, None)
    assert st == 1  # misaligned dh


def test_selftest_rejects_invalid_arguments(L):
    c = ctypes.c_void_p
    assert L.fkl_selftest_gemm(c(16), c(16), c(16), 12, 16, 16, 0, 0, 256, c(16), None) == 1
    assert L.fkl_selftest_gemm(c(16), c(16), c(16), 16, 16, 16, 2, 0, 256, c(16), None) == 1
    assert L.fkl_selftest_gemm(c(16), c(16), c(16), 16, 16, 16, 0, 0, 64, c(16), None) == 1
