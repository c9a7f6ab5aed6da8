"""The KL + hard-label cross-entropy mixture (fkl_mix_forward / fkl_mix_backward)
against the fp64 oracle, and against the plain loss at alpha = 1."""
import numpy as np
import pytest
import torch

import oracle
from lm_head_kl_fkl_b300 import api, synth
from tests.gpu_helpers import (TOL_GRAD_REL_L2, TOL_LOSS_REL, TOL_LSE_ABS, both_oracles, oracle_inputs,
                               rel_l2, run_fused, to_device)

pytestmark = pytest.mark.gpu


def _labels(x, seed):
    return np.random.default_rng(seed).integers(0, x["V"], x["N"]).astype(np.int32)


def _run_mix(xd, label, alpha, chunk=0, grad=None):
    lab = torch.from_numpy(label).to(xd["h"].device)
    loss, lse, lse1 = api.mix_forward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], lab, xd["T"], alpha,
                                      chunk)
    g = None if grad is None else torch.tensor([grad], dtype=torch.float32, device=xd["h"].device)
    dh, dW = api.mix_backward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], lab, xd["T"], alpha, lse, lse1,
                              grad_loss=g, chunk=chunk)
    torch.cuda.synchronize()
    return dict(loss=float(loss.item()), lse=lse.cpu().numpy().astype(np.float64),
                lse1=lse1.cpu().numpy().astype(np.float64), dh=dh.float().cpu().numpy().astype(np.float64),
                dW=dW.cpu().numpy().astype(np.float64))


def _check(x, label, alpha, out, grad=1.0, oracles=None):
    """Against the plain C++ and the numpy fp64 oracles (or the ones given)."""
    h, W = oracle_inputs(x)
    for name, orc in (oracles or both_oracles()):
        ref = orc.forward_mix(h, W, x["idx"], x["t"], x["mask"], label, x["T"], alpha)
        g = orc.backward_mix(h, W, x["idx"], x["t"], x["mask"], label, x["T"], alpha, grad_loss=grad)
        assert abs(out["loss"] - ref["loss"]) <= TOL_LOSS_REL * abs(ref["loss"]), (name, out["loss"], ref["loss"])
        assert np.abs(out["lse"] - ref["lse"]).max() <= TOL_LSE_ABS, name
        assert np.abs(out["lse1"] - ref["lse1"]).max() <= TOL_LSE_ABS, name
        assert rel_l2(out["dh"], g["dh"]) <= TOL_GRAD_REL_L2, (name, rel_l2(out["dh"], g["dh"]))
        assert rel_l2(out["dW"], g["dW"]) <= TOL_GRAD_REL_L2, (name, rel_l2(out["dW"], g["dW"]))


CASES = [
    # N, d, V, K, T, index, chunk, alpha
    (300, 136, 1000, 16, 2.0, "uniform", 128, 0.5),
    (257, 64, 1001, 8, 1.0, "uniform", 0, 0.3),
    (640, 256, 4096, 100, 3.0, "zipf1.1", 256, 0.9),
    (96, 200, 777, 5, 1.0, "half-student", 0, 0.0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "N{}_T{}_a{}".format(c[0], c[4], c[7]))
def test_mixture_parity(case):
    N, d, V, K, T, index, chunk, alpha = case
    x = synth.make_inputs(N, d, V, K, T, 0.05, index, seed=8000 + N)
    label = _labels(x, 8100 + N)
    _check(x, label, alpha, _run_mix(to_device(x), label, alpha, chunk, grad=1.25), grad=1.25)


def test_alpha_one_is_the_plain_loss():
    x = synth.make_inputs(400, 128, 2000, 20, 2.0, 0.05, "uniform", seed=8200)
    xd = to_device(x)
    mix = _run_mix(xd, _labels(x, 8201), 1.0)
    plain = run_fused(xd)
    assert mix["loss"] == plain["loss"]
    assert np.array_equal(mix["lse"], plain["lse"])
    assert rel_l2(mix["dh"], plain["dh"]) <= 1e-3 and rel_l2(mix["dW"], plain["dW"]) <= 1e-4


def test_label_out_of_range_sets_status():
    x = synth.make_inputs(64, 64, 300, 4, 1.0, 0.0, "uniform", seed=8300)
    label = _labels(x, 8301)
    label[5] = 300
    xd = to_device(x)
    ws = api.alloc_workspace(64, 64, 300, 4)
    api.mix_forward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], torch.from_numpy(label).cuda(), 1.0, 0.5,
                    ws=ws)
    assert api.get_status(ws) == 3


def test_small_lm_head_workload():
    """The small LM head workload (N=4096, d=2048, V=32768, K=100, T=2) at full size."""
    x = synth.config_inputs(1)
    label = _labels(x, 8400)
    _check(x, label, 0.5, _run_mix(to_device(x), label, 0.5), oracles=[("numpy", oracle)])
