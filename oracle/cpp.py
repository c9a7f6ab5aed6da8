"""ctypes front of the plain C++ fp64 oracle (``fkl_oracle.cpp``).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``.  The functions mirror
the numpy oracle's names and signatures so that the same pins run on both; all
arithmetic happens in the C++ source, this module only converts arrays and
passes pointers.

The library is compiled with g++ (``-O2``, no fast-math: every sum keeps the
source's order) into ``oracle/libfkl_oracle.so`` by :func:`build`, which
``__graft_entry__.build()`` calls; :func:`load` rebuilds it when the source is
newer.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fkl_oracle.cpp")
LIB = os.path.join(HERE, "libfkl_oracle.so")

_lock = threading.Lock()
_default = None

_d = ctypes.POINTER(ctypes.c_double)
_i32 = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u8 = ctypes.POINTER(ctypes.c_uint8)
_I, _L, _F = ctypes.c_int, ctypes.c_int64, ctypes.c_double

_SIGS = {
    "fklo_teacher": [_d, _L, _L, _F, _d, _u8],
    "fklo_forward": [_d, _d, _i32, _d, _u8, _L, _L, _L, _L, _F, _I, _d, _d, _u8, _d, _i64p],
    "fklo_backward": [_d, _d, _i32, _d, _u8, _L, _L, _L, _L, _F, _F, _L, _I, _d, _d],
    "fklo_rows": [_d, _d, _i32, _d, _u8, _L, _L, _L, _L, _F, _F, _i64p, _L, _I, _d, _d, _d, _i64p],
    "fklo_dW_rows": [_d, _d, _i32, _d, _u8, _L, _L, _L, _L, _F, _F, _d, _i64p, _L, _I, _d],
    "fklo_student_lse": [_d, _d, _L, _L, _L, _F, _I, _d],
    "fklo_teacher_topk": [_d, _d, _L, _L, _L, _L, _I, _i64p, _d],
    "fklo_forward_mix": [_d, _d, _i32, _d, _u8, _i32, _L, _L, _L, _L, _F, _F, _I, _d, _d, _d, _d, _u8, _d, _i64p],
    "fklo_backward_mix": [_d, _d, _i32, _d, _u8, _i32, _L, _L, _L, _L, _F, _F, _F, _I, _d, _d],
}


def compile_library(src: str, out: str) -> str:
    """g++ -O2 -shared of one oracle source file."""
    cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", "-o", out, src]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"g++ failed on {src}:\n{r.stderr}")
    return out


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        compile_library(SRC, LIB)
    return LIB


def threads() -> int:
    """Worker threads per call: FKL_ORACLE_THREADS, else every host core."""
    return int(os.environ.get("FKL_ORACLE_THREADS", "0")) or (os.cpu_count() or 1)


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a, typ):
    return a.ctypes.data_as(typ)


class CppOracle:
    """The C++ oracle behind one shared library (the default, or a test's mutant)."""

    def __init__(self, path: str):
        self.path = path
        self.lib = ctypes.CDLL(path)
        for name, args in _SIGS.items():
            f = getattr(self.lib, name)
            f.restype = None
            f.argtypes = args

    # -- marshalling helpers
    @staticmethod
    def _common(h, W, idx, tlogit, mask):
        h, W, t = _f64(h), _f64(W), _f64(tlogit)
        idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int32))
        m = None if mask is None else np.ascontiguousarray(np.asarray(mask) != 0, dtype=np.uint8)
        return h, W, idx, t, m

    def teacher_distribution(self, tlogit, T):
        t = _f64(tlogit)
        N, K = t.shape
        p = np.empty((N, K))
        ok = np.empty(N, dtype=np.uint8)
        self.lib.fklo_teacher(_p(t, _d), N, K, float(T), _p(p, _d), _p(ok, _u8))
        return p, ok.astype(bool)

    def forward(self, h, W, idx, tlogit, mask, T, row_block=256):
        del row_block  # the C++ oracle takes rows one at a time; no blocking to choose
        h, W, idx, t, m = self._common(h, W, idx, tlogit, mask)
        N, d = h.shape
        V, K = W.shape[0], idx.shape[1]
        lse, kl = np.empty(N), np.empty(N)
        valid = np.empty(N, dtype=np.uint8)
        loss = ctypes.c_double()
        nv = ctypes.c_int64()
        self.lib.fklo_forward(_p(h, _d), _p(W, _d), _p(idx, _i32), _p(t, _d), None if m is None else _p(m, _u8),
                              N, d, V, K, float(T), threads(), _p(lse, _d), _p(kl, _d), _p(valid, _u8),
                              ctypes.byref(loss), ctypes.byref(nv))
        return dict(loss=loss.value, lse=lse, kl=kl, n_valid=int(nv.value), valid=valid.astype(bool))

    def backward(self, h, W, idx, tlogit, mask, T, grad_loss=1.0, row_block=256):
        h, W, idx, t, m = self._common(h, W, idx, tlogit, mask)
        N, d = h.shape
        V, K = W.shape[0], idx.shape[1]
        dh, dW = np.empty((N, d)), np.empty((V, d))
        self.lib.fklo_backward(_p(h, _d), _p(W, _d), _p(idx, _i32), _p(t, _d), None if m is None else _p(m, _u8),
                               N, d, V, K, float(T), float(grad_loss), int(row_block), threads(),
                               _p(dh, _d), _p(dW, _d))
        return dict(dh=dh, dW=dW)

    def rows_forward_backward(self, h, W, idx, tlogit, mask, T, rows, grad_loss=1.0, row_block=128):
        del row_block
        h, W, idx, t, m = self._common(h, W, idx, tlogit, mask)
        N, d = h.shape
        V, K = W.shape[0], idx.shape[1]
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = len(rows)
        lse, kl, dh = np.empty(n), np.empty(n), np.empty((n, d))
        nv = ctypes.c_int64()
        self.lib.fklo_rows(_p(h, _d), _p(W, _d), _p(idx, _i32), _p(t, _d), None if m is None else _p(m, _u8),
                           N, d, V, K, float(T), float(grad_loss), _p(rows, _i64p), n, threads(),
                           _p(lse, _d), _p(kl, _d), _p(dh, _d), ctypes.byref(nv))
        return dict(lse=lse, kl=kl, dh=dh, n_valid=int(nv.value))

    def dW_rows(self, h, W, idx, tlogit, mask, T, lse, vocab_rows, grad_loss=1.0, row_block=4096):
        del row_block
        h, W, idx, t, m = self._common(h, W, idx, tlogit, mask)
        N, d = h.shape
        V, K = W.shape[0], idx.shape[1]
        lse = _f64(lse)
        vr = np.ascontiguousarray(np.asarray(vocab_rows, dtype=np.int64))
        out = np.empty((len(vr), d))
        self.lib.fklo_dW_rows(_p(h, _d), _p(W, _d), _p(idx, _i32), _p(t, _d), None if m is None else _p(m, _u8),
                              N, d, V, K, float(T), float(grad_loss), _p(lse, _d), _p(vr, _i64p), len(vr),
                              threads(), _p(out, _d))
        return out

    def student_lse(self, h, W, T, row_block=256):
        del row_block
        h, W = _f64(h), _f64(W)
        N, d = h.shape
        out = np.empty(N)
        self.lib.fklo_student_lse(_p(h, _d), _p(W, _d), N, d, W.shape[0], float(T), threads(), _p(out, _d))
        return out


def _teacher_topk(self, h, W, K, rows=None, row_block=256):
    """Per row the K largest logits (descending, ties by ascending id): (idx, logit, None)."""
    del row_block
    h, W = _f64(h), _f64(W)
    if rows is not None:
        h = np.ascontiguousarray(h[np.asarray(rows, dtype=np.int64)])
    N, d = h.shape
    V = W.shape[0]
    idx = np.empty((N, K), dtype=np.int64)
    val = np.empty((N, K))
    self.lib.fklo_teacher_topk(_p(h, _d), _p(W, _d), N, d, V, int(K), threads(), _p(idx, _i64p), _p(val, _d))
    return idx, val, None


CppOracle.teacher_topk = _teacher_topk


def _forward_mix(self, h, W, idx, tlogit, mask, label, T, alpha, row_block=256):
    """KL + hard-label cross-entropy mixture: the forward's dict plus lse1 and ce."""
    del row_block
    h, W, idx, t, m = self._common(h, W, idx, tlogit, mask)
    lab = np.ascontiguousarray(np.asarray(label, dtype=np.int32))
    N, d = h.shape
    V, K = W.shape[0], idx.shape[1]
    lse, lse1, kl, ce = (np.empty(N) for _ in range(4))
    valid = np.empty(N, dtype=np.uint8)
    loss = ctypes.c_double()
    nv = ctypes.c_int64()
    self.lib.fklo_forward_mix(_p(h, _d), _p(W, _d), _p(idx, _i32), _p(t, _d), None if m is None else _p(m, _u8),
                              _p(lab, _i32), N, d, V, K, float(T), float(alpha), threads(), _p(lse, _d),
                              _p(lse1, _d), _p(kl, _d), _p(ce, _d), _p(valid, _u8), ctypes.byref(loss),
                              ctypes.byref(nv))
    return dict(loss=loss.value, lse=lse, lse1=lse1, kl=kl, ce=ce, n_valid=int(nv.value), valid=valid.astype(bool))


def _backward_mix(self, h, W, idx, tlogit, mask, label, T, alpha, grad_loss=1.0, row_block=256):
    """dh, dW of the mixture times grad_loss."""
    del row_block
    h, W, idx, t, m = self._common(h, W, idx, tlogit, mask)
    lab = np.ascontiguousarray(np.asarray(label, dtype=np.int32))
    N, d = h.shape
    V, K = W.shape[0], idx.shape[1]
    dh, dW = np.empty((N, d)), np.empty((V, d))
    self.lib.fklo_backward_mix(_p(h, _d), _p(W, _d), _p(idx, _i32), _p(t, _d), None if m is None else _p(m, _u8),
                               _p(lab, _i32), N, d, V, K, float(T), float(alpha), float(grad_loss), threads(),
                               _p(dh, _d), _p(dW, _d))
    return dict(dh=dh, dW=dW)


CppOracle.forward_mix = _forward_mix
CppOracle.backward_mix = _backward_mix


def load() -> CppOracle:
    """The default C++ oracle (compiled on first use if missing or stale)."""
    global _default
    with _lock:
        if _default is None:
            _default = CppOracle(build())
    return _default
