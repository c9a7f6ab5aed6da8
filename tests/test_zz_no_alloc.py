"""fkl_forward_noalloc: the forward for callers that cannot allocate device memory.

Some callers own no device allocator (a plain C host program, or a plug-in inside
a runtime that has already reserved the GPU's memory for its own pool), and some
step loops must not call cudaMalloc/cudaFree, which can synchronise the device
and can fail under memory pressure.  For them the library carries a fixed
64 MiB scratch array of its own; the caller passes only inputs and outputs.

Checked here through the C ABI: two calls in a row (different sizes, so the
second one runs over the first one's leftovers in the shared scratch) give
bit for bit the loss and lse of fkl_forward on a caller workspace (the same
kernels in the same order), and the first of them matches the fp64 oracle
within the parity tolerances; a teacher id outside [0, V) is reported through
the status output; a size whose scratch would exceed the array is refused on the
host before any launch.

This file is collected last on purpose (its name sorts after every other test).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from lm_head_kl_fkl_b300 import _lib, api, synth
from tests.gpu_helpers import TOL_LOSS_REL, TOL_LSE_ABS, oracle_inputs, to_device

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 << 20


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(xd, chunk=0):
    """One call of fkl_forward_noalloc; returns (status, loss, lse, device status)."""
    h, W, idx = xd["h"], xd["W"], xd["idx"]
    N, d = h.shape
    V, K = W.shape[0], idx.shape[1]
    dev = h.device
    loss = torch.full((1,), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((N,), float("nan"), dtype=torch.float32, device=dev)
    dstat = torch.full((1,), -1, dtype=torch.int32, device=dev)
    st = _lib.lib().fkl_forward_noalloc(
        _p(h), _p(W), _p(idx), _p(xd["t"]), _p(xd["mask"]), N, d, V, K, ctypes.c_float(xd["T"]), chunk,
        _p(loss), _p(lse), _p(dstat), ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    torch.cuda.synchronize()
    return st, loss, lse, int(dstat.item())


def _check_against_workspace_forward(xd, chunk, out):
    st, loss, lse, dstat = out
    assert st == 0, _lib.lib().fkl_last_error().decode()
    assert dstat == 0
    ref_loss, ref_lse = api.forward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], xd["T"], chunk)
    torch.cuda.synchronize()
    # the same launch sequence on the same inputs: bit-identical results
    assert float(loss.item()) == float(ref_loss.item()), (float(loss.item()), float(ref_loss.item()))
    assert torch.equal(lse, ref_lse), float((lse - ref_lse).abs().max().item())


def _check_against_oracle(x, out):
    _, loss, lse, _ = out
    h, W = oracle_inputs(x)
    ref = oracle.forward(h, W, x["idx"], x["t"], x["mask"], x["T"])
    assert abs(float(loss.item()) - ref["loss"]) <= TOL_LOSS_REL * abs(ref["loss"]), (float(loss.item()), ref["loss"])
    err = float(np.abs(lse.cpu().numpy().astype(np.float64) - ref["lse"]).max())
    assert err <= TOL_LSE_ABS, err


def test_two_calls_match_workspace_forward():
    # first call: several chunks and vocabulary tiles, ragged everywhere
    xa = synth.make_inputs(700, 136, 3001, 24, 1.5, 0.05, "uniform", seed=4242)
    da = to_device(xa)
    out_a = _noalloc(da, chunk=256)
    _check_against_workspace_forward(da, 256, out_a)
    _check_against_oracle(xa, out_a)
    # second call, straight after: other sizes and the default chunk, over the
    # scratch contents the first call left behind
    xb = synth.make_inputs(1300, 256, 5000, 100, 1.0, 0.05, "zipf1.1", seed=4243)
    db = to_device(xb)
    _check_against_workspace_forward(db, 0, _noalloc(db))


def test_bad_teacher_id_reported_in_status():
    x = synth.make_inputs(64, 64, 300, 4, 1.0, 0.0, "uniform", seed=4244)
    x["idx"][7, 2] = 300  # == V
    st, _, _, dstat = _noalloc(to_device(x))
    assert st == 0 and dstat == 3  # FKL_ERR_INDEX
    x["idx"][7, 2] = 0 if 0 not in x["idx"][7] else 299
    st, _, _, dstat = _noalloc(to_device(x))
    assert st == 0 and dstat == 0  # the header is cleared on every call


def test_oversized_request_refused_before_launch():
    # V = 201088 at chunk 8192 needs 12 * 8192 * 786 bytes of partials alone (> 64 MiB)
    dev = torch.device("cuda")
    tiny = torch.zeros(64, dtype=torch.bfloat16, device=dev)
    ids = torch.zeros(8, dtype=torch.int32, device=dev)
    tl = torch.zeros(8, dtype=torch.float32, device=dev)
    out = torch.zeros(8, dtype=torch.float32, device=dev)
    before = api.launch_count()
    st = _lib.lib().fkl_forward_noalloc(_p(tiny), _p(tiny), _p(ids), _p(tl), None, 8192, 2880, 201088, 100,
                                        ctypes.c_float(1.0), 8192, _p(out), _p(out), None, None)
    assert st == 2  # FKL_ERR_WORKSPACE
    msg = _lib.lib().fkl_last_error().decode()
    assert "scratch" in msg and str(SCRATCH_BYTES) in msg
    assert api.launch_count() == before

