"""The torch layer on a GPU: caller-supplied outputs and workspaces of the wrong
kind are refused with a Python error before any launch; a workspace of any dtype
is sized in bytes; the autograd loss raises on a device-side error when asked to."""
import numpy as np
import pytest
import torch

from lm_head_kl_fkl_b300 import api, synth
from tests.gpu_helpers import to_device

pytestmark = pytest.mark.gpu


def _x(seed=5100):
    return to_device(synth.make_inputs(96, 64, 500, 8, 1.0, 0.05, "uniform", seed=seed))


@pytest.mark.parametrize("kw", [
    dict(lse=lambda d: torch.empty(95, dtype=torch.float32, device=d)),
    dict(lse=lambda d: torch.empty(96, dtype=torch.float16, device=d)),
    dict(loss=lambda d: torch.empty(2, dtype=torch.float32, device=d)),
    dict(ws=lambda d: torch.empty(1 << 20, dtype=torch.uint8)),            # host memory
])
def test_forward_refuses_wrong_outputs(kw):
    xd = _x()
    dev = xd["h"].device
    args = {k: f(dev) for k, f in kw.items()}
    before = api.launch_count()
    with pytest.raises((ValueError, TypeError)):
        api.forward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], 1.0, **args)
    assert api.launch_count() == before


@pytest.mark.parametrize("kw", [
    dict(dh=lambda d: torch.empty((96, 64), dtype=torch.float32, device=d)),
    dict(dW=lambda d: torch.empty((499, 64), dtype=torch.float32, device=d)),
    dict(dW=lambda d: torch.empty((64, 500), dtype=torch.float32, device=d).t()),  # not contiguous
])
def test_backward_refuses_wrong_outputs(kw):
    xd = _x()
    dev = xd["h"].device
    _, lse = api.forward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], 1.0)
    args = {k: f(dev) for k, f in kw.items()}
    before = api.launch_count()
    with pytest.raises((ValueError, TypeError)):
        api.backward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], 1.0, lse, **args)
    assert api.launch_count() == before


def test_workspace_of_any_dtype_is_sized_in_bytes():
    xd = _x()
    need = api.workspace_size(96, 64, 500, 8)
    ws32 = torch.empty((need + 3) // 4, dtype=torch.float32, device=xd["h"].device)
    loss, lse = api.forward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], 1.0, ws=ws32)
    ref_loss, ref_lse = api.forward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], 1.0)
    assert loss.item() == ref_loss.item() and torch.equal(lse, ref_lse)
    small = torch.empty(need // 4 - 1, dtype=torch.float32, device=xd["h"].device)  # < need bytes
    with pytest.raises(api.FKLError):
        api.forward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], 1.0, ws=small)


@pytest.mark.parametrize("keep_logits", [False, True])
def test_autograd_check_status_raises_on_bad_teacher_id(keep_logits):
    x = synth.make_inputs(96, 64, 500, 8, 1.0, 0.0, "uniform", seed=5101)
    x["idx"][3, 1] = 500  # == V
    xd = to_device(x)
    h = xd["h"].clone().requires_grad_(True)
    W = xd["W"].clone().requires_grad_(True)
    with pytest.raises(api.FKLError, match="FKL_ERR_INDEX"):
        api.fkl_loss(h, W, xd["idx"], xd["t"], xd["mask"], 1.0, keep_logits=keep_logits, check_status=True)
    # a valid id passes through the same checks
    x["idx"][3, 1] = 0 if 0 not in x["idx"][3] else 499
    xd = to_device(x)
    loss = api.fkl_loss(h, W, xd["idx"], xd["t"], xd["mask"], 1.0, keep_logits=keep_logits, check_status=True)
    loss.backward()
    assert np.isfinite(loss.item()) and torch.isfinite(h.grad.float()).all()
