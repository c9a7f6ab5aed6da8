"""Host-side argument checks of every loss, producer and helper entry point of
libfkl.so: each rejection below is decided before any CUDA call, so these run on a
machine without a GPU.  The pointers are plain integers that are never dereferenced
(16 is 16-byte aligned, 24 is not)."""
import ctypes

import pytest

from lm_head_kl_fkl_b300 import _lib

INVALID, WORKSPACE = 1, 2
P = ctypes.c_void_p
A16, A24 = P(16), P(24)
BIG = 1 << 40


@pytest.fixture(scope="module")
def L():
    import os
    if not os.path.exists(_lib.LIB_PATH):
        from lm_head_kl_fkl_b300 import build
        build.build(quiet=True)
    return _lib.lib()


def test_size_limits_give_zero_workspace(L):
    ws = L.fkl_workspace_size
    assert ws(100, 65536, 1000, 8, 0) > 0
    for args in [(100, 65544, 1000, 8, 0),          # d above 65536
                 (100, 64, (1 << 30) + 1, 8, 0),    # V above 2^30
                 (100, 64, 1000, 8, (1 << 20) + 128),  # chunk above 2^20
                 ((1 << 40) + 1, 64, 1000, 8, 0)]:  # N above 2^40
        assert ws(*args) == 0, args
        assert L.fkl_topk_workspace_size(*args) == 0, args


def _mix_fwd(L, label=A16, alpha=0.5, ws_bytes=BIG, lse1=A16):
    return L.fkl_mix_forward(A16, A16, A16, A16, None, label, 10, 64, 100, 4, 1.0, alpha, 0,
                             A16, A16, lse1, A16, ws_bytes, None)


def _mix_bwd(L, label=A16, alpha=0.5, dh=A16, ws_bytes=BIG):
    return L.fkl_mix_backward(A16, A16, A16, A16, None, label, 10, 64, 100, 4, 1.0, alpha, 0,
                              A16, A16, None, dh, A16, A16, ws_bytes, None)


@pytest.mark.parametrize("kw", [dict(label=None), dict(lse1=None), dict(alpha=-0.1), dict(alpha=1.5),
                                dict(alpha=float("nan"))])
def test_mix_forward_rejects(L, kw):
    assert _mix_fwd(L, **kw) == INVALID
    assert L.fkl_last_error().decode()


def test_mix_forward_small_workspace(L):
    assert _mix_fwd(L, ws_bytes=1000) == WORKSPACE


@pytest.mark.parametrize("kw", [dict(label=None), dict(alpha=2.0), dict(dh=None), dict(dh=A24)])
def test_mix_backward_rejects(L, kw):
    assert _mix_bwd(L, **kw) == INVALID


def _fb(L, dh=A16, dW=A16, loss=A16, ws_bytes=BIG, chunk=0, K=4):
    return L.fkl_forward_backward(A16, A16, A16, A16, None, 10, 64, 100, K, 1.0, chunk, None, loss, A16,
                                  dh, dW, A16, ws_bytes, None)


@pytest.mark.parametrize("kw", [dict(dh=None), dict(dW=None), dict(loss=None), dict(dW=A24),
                                dict(chunk=64), dict(K=0)])
def test_forward_backward_rejects(L, kw):
    assert _fb(L, **kw) == INVALID


def test_forward_backward_small_workspace(L):
    assert _fb(L, ws_bytes=1 << 10) == WORKSPACE
    assert b"needed" in L.fkl_last_error()


def _topk(L, h=A16, idx=A16, K=4, V=100, ws=A16, ws_bytes=BIG):
    return L.fkl_teacher_topk(h, A16, 10, 64, V, K, 0, idx, A16, ws, ws_bytes, None)


@pytest.mark.parametrize("kw", [dict(h=None), dict(idx=None), dict(ws=None), dict(K=0), dict(K=257),
                                dict(K=8, V=7), dict(h=A24)])
def test_teacher_topk_rejects(L, kw):
    assert _topk(L, **kw) == INVALID


def test_teacher_topk_small_workspace(L):
    assert _topk(L, ws_bytes=1 << 10) == WORKSPACE


@pytest.mark.parametrize("args", [
    (None, A16, 10, 64, 100, A16),   # null dh
    (A16, A16, 10, 64, 100, None),   # null grad
    (A16, A16, 0, 64, 100, A16),     # N = 0
    (A16, A16, 10, 60, 100, A16),    # d not a multiple of 8
    (A24, A16, 10, 64, 100, A16),    # misaligned dh
])
def test_scale_grads_rejects(L, args):
    assert L.fkl_scale_grads(*args, None) == INVALID


def test_noalloc_refuses_sizes_beyond_its_scratch(L):
    # 2^24 rows: the 4 bytes per row alone exceed the scratch, so no chunk fits and N is named
    st = L.fkl_forward_noalloc(A16, A16, A16, A16, None, 1 << 24, 2880, 201088, 100, 1.0, 0,
                               A16, A16, None, None)
    assert st == WORKSPACE
    msg = L.fkl_last_error()
    assert b"scratch" in msg and b"smallest chunk" in msg and b"fewer rows" in msg
    # a size that fits at a smaller chunk: the message asks for one
    st = L.fkl_forward_noalloc(A16, A16, A16, A16, None, 32768, 2880, 201088, 100, 1.0, 8192,
                               A16, A16, None, None)
    assert st == WORKSPACE
    assert b"smaller chunk" in L.fkl_last_error()
    # and the usual argument checks come first
    st = L.fkl_forward_noalloc(A16, A16, A16, A16, None, 10, 60, 100, 4, 1.0, 0, A16, A16, None, None)
    assert st == INVALID


def test_status_and_selftest_entries_reject(L):
    assert L.fkl_get_status(None, None) == INVALID
    assert L.fkl_selftest_wait_timeout(None, 10_000, None) == INVALID
    assert L.fkl_selftest_wait_timeout(A16, 10, None) == INVALID
    assert L.fkl_selftest_wait_timeout(A16, 3_000_000_000, None) == INVALID


def test_last_error_is_per_thread(L):
    import threading
    assert _fb(L, dh=None) == INVALID
    main_msg = L.fkl_last_error().decode()
    seen = {}

    def other():
        seen["before"] = L.fkl_last_error().decode()
        assert _topk(L, K=0) == INVALID
        seen["after"] = L.fkl_last_error().decode()

    t = threading.Thread(target=other)
    t.start()
    t.join()
    assert seen["before"] == ""
    assert seen["after"] and seen["after"] != main_msg
    assert L.fkl_last_error().decode() == main_msg
