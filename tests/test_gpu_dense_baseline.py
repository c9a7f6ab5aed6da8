"""The dense comparison baseline of bench.py (full N x V logits in plain torch) computes
the same loss and gradients as the fp64 oracle, so that its memory and time are those
of the same problem."""
import os
import sys

import numpy as np
import pytest
import torch

import oracle
from lm_head_kl_fkl_b300 import synth
from tests.gpu_helpers import TOL_GRAD_REL_L2, TOL_LOSS_REL, oracle_inputs, rel_l2, to_device

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [1.0, 2.0])
def test_dense_baseline_matches_oracle(T):
    x = synth.make_inputs(300, 128, 3000, 16, T, 0.05, "uniform", seed=9500)
    x["t"][4, 3:] = -np.inf  # entries without mass
    xd = to_device(x)
    loss, dh, dW = bench.dense_kl_step(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], T)
    h, W = oracle_inputs(x)
    ref = oracle.forward(h, W, x["idx"], x["t"], x["mask"], T)
    g = oracle.backward(h, W, x["idx"], x["t"], x["mask"], T)
    assert abs(loss.item() - ref["loss"]) <= TOL_LOSS_REL * abs(ref["loss"])
    assert rel_l2(dh.double().cpu().numpy(), g["dh"]) <= TOL_GRAD_REL_L2
    assert rel_l2(dW.double().cpu().numpy(), g["dW"]) <= TOL_GRAD_REL_L2
