"""Failure detection on the GPU without a fault: a pipeline wait that nothing
completes gives up after its limit, the status word says FKL_ERR_TIMEOUT, and the
context stays usable for the next call."""
import ctypes

import numpy as np
import pytest
import torch

from lm_head_kl_fkl_b300 import _lib, api, synth
from tests.gpu_helpers import run_fused, to_device

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    assert _lib.lib().fkl_selftest_wait_timeout(ctypes.c_void_p(ws.data_ptr()), 20_000_000, stream) == 0
    e1.record()
    assert api.get_status(ws) == 6  # FKL_ERR_TIMEOUT
    assert e0.elapsed_time(e1) >= 19.0  # it waited (about) the whole limit, then returned

    # the context is intact: a normal call on the same workspace succeeds and clears the word
    x = synth.make_inputs(200, 64, 500, 8, 1.0, 0.05, "uniform", seed=9300)
    xd = to_device(x)
    big = api.alloc_workspace(200, 64, 500, 8)
    loss, _ = api.forward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], 1.0, ws=big)
    assert api.get_status(big) == 0 and np.isfinite(loss.item())
    out = run_fused(xd)
    assert np.isfinite(out["dW"]).all()


def test_selftest_rejects_bad_arguments():
    L = _lib.lib()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert L.fkl_selftest_wait_timeout(None, 20_000_000, None) == 1
    assert L.fkl_selftest_wait_timeout(ctypes.c_void_p(ws.data_ptr()), 10, None) == 1
    assert L.fkl_selftest_wait_timeout(ctypes.c_void_p(ws.data_ptr()), 5_000_000_000, None) == 1
