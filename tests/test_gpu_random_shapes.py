"""Seeded random shapes within the library's limits: the two-call path and the
one-call path against the fp64 oracles, element by element.  Sizes are drawn so that
the plain C++ oracle finishes each case in a few seconds (N d V <= 4e9)."""
import numpy as np
import pytest
import torch

from lm_head_kl_fkl_b300 import api, synth
from tests.gpu_helpers import (TOL_GRAD_REL_L2, TOL_LOSS_REL, TOL_LSE_ABS, both_oracles, oracle_inputs, rel_l2,
                               run_fused, to_device)

pytestmark = pytest.mark.gpu


def _shape(i):
    rng = np.random.default_rng(12000 + i)
    while True:
        N = int(rng.integers(1, 1600))
        d = 8 * int(rng.integers(1, 129))
        V = int(rng.integers(8, 24000))
        K = int(min(V, rng.integers(1, 257)))
        if N * d * V <= 4e9:
            break
    T = float(np.exp(rng.uniform(np.log(0.25), np.log(4.0))))
    chunk = int(rng.choice([0, 128, 256, 384, 640]))
    pad = float(rng.uniform(0.0, 0.2))
    index = str(rng.choice(["uniform", "zipf1.1"]))
    return N, d, V, K, T, chunk, pad, index


CASES = [_shape(i) for i in range(12)]


def _check(x, out, name_prefix=""):
    h, W = oracle_inputs(x)
    for name, orc in both_oracles():
        ref = orc.forward(h, W, x["idx"], x["t"], x["mask"], x["T"])
        g = orc.backward(h, W, x["idx"], x["t"], x["mask"], x["T"])
        tag = name_prefix + name
        if ref["n_valid"] > 0:
            assert abs(out["loss"] - ref["loss"]) <= TOL_LOSS_REL * abs(ref["loss"]), (tag, out["loss"], ref["loss"])
            assert rel_l2(out["dh"], g["dh"]) <= TOL_GRAD_REL_L2, (tag, rel_l2(out["dh"], g["dh"]))
            assert rel_l2(out["dW"], g["dW"]) <= TOL_GRAD_REL_L2, (tag, rel_l2(out["dW"], g["dW"]))
        else:
            assert out["loss"] == 0.0 and not out["dh"].any() and not out["dW"].any(), tag
        assert np.abs(out["lse"] - ref["lse"]).max() <= TOL_LSE_ABS, tag


@pytest.mark.parametrize("case", CASES, ids=lambda c: "N{}_d{}_V{}_K{}_T{:.2f}_c{}".format(*c[:6]))
def test_random_shape_two_call_and_one_call(case):
    N, d, V, K, T, chunk, pad, index = case
    x = synth.make_inputs(N, d, V, K, T, pad, index, seed=12500 + N + V)
    xd = to_device(x)
    _check(x, run_fused(xd, chunk=chunk), "two-call/")
    loss, lse, dh, dW = api.forward_backward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], T, chunk=chunk)
    torch.cuda.synchronize()
    one = dict(loss=float(loss.item()), lse=lse.cpu().numpy().astype(np.float64),
               dh=dh.float().cpu().numpy().astype(np.float64), dW=dW.cpu().numpy().astype(np.float64))
    _check(x, one, "one-call/")


def _mix_shape(i):
    rng = np.random.default_rng(13000 + i)
    while True:
        N = int(rng.integers(1, 1200))
        d = 8 * int(rng.integers(1, 97))
        V = int(rng.integers(8, 16000))
        K = int(min(V, rng.integers(1, 257)))
        if N * d * V <= 2e9:
            break
    T = float(np.exp(rng.uniform(np.log(0.5), np.log(4.0))))
    chunk = int(rng.choice([0, 128, 256, 512]))
    alpha = float(rng.choice([0.0, 0.25, 0.5, 0.9, 1.0]))
    return N, d, V, K, T, chunk, alpha


MIX_CASES = [_mix_shape(i) for i in range(6)]


@pytest.mark.parametrize("case", MIX_CASES, ids=lambda c: "N{}_d{}_V{}_K{}_T{:.2f}_c{}_a{}".format(*c))
def test_random_shape_mixture(case):
    """The KL + hard-label cross-entropy mixture on seeded random shapes, labels and
    alpha, against both fp64 oracles."""
    from tests.test_gpu_mixture import _check as mix_check, _labels, _run_mix
    N, d, V, K, T, chunk, alpha = case
    x = synth.make_inputs(N, d, V, K, T, 0.05, "uniform", seed=13500 + N + V)
    label = _labels(x, 13600 + N)
    mix_check(x, label, alpha, _run_mix(to_device(x), label, alpha, chunk, grad=0.75), grad=0.75)


def _topk_shape(i):
    rng = np.random.default_rng(14000 + i)
    while True:
        N = int(rng.integers(1, 900))
        d = 8 * int(rng.integers(1, 65))
        V = int(rng.integers(1, 60000))
        K = int(min(V, rng.integers(1, 257)))
        if N * d * V <= 2e9:
            break
    chunk = int(rng.choice([0, 128, 256, 384]))
    return N, d, V, K, chunk


TOPK_CASES = [_topk_shape(i) for i in range(8)]


@pytest.mark.parametrize("case", TOPK_CASES, ids=lambda c: "N{}_d{}_V{}_K{}_c{}".format(*c))
def test_random_shape_teacher_topk(case):
    """The teacher top-K cache producer on seeded random shapes and chunk sizes, checked
    as the dedicated top-K tests check it: what is unique exactly, the rest for validity."""
    from tests.test_gpu_teacher_topk import _bf16, _check as topk_check, _run
    N, d, V, K, chunk = case
    rng = np.random.default_rng(14500 + N + V)
    h = _bf16(rng.standard_normal((N, d)))
    W = _bf16(rng.standard_normal((V, d)) / np.sqrt(d))
    idx, val = _run(h, W, K, chunk)
    topk_check(h, W, K, idx, val)
