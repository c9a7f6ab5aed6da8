"""Fused CUDA path against the fp64 oracles, element by element, on sizes the
oracles finish in seconds (several tiles, ragged tails in N, d and V, several
chunks), plus edge cases.  Every case is compared with both independent oracles:
the plain C++ one (loops, one full logit row per token) and the numpy one."""
import numpy as np
import pytest
import torch

import oracle
from lm_head_kl_fkl_b300 import api, synth
from tests.gpu_helpers import (TOL_GRAD_REL_L2, TOL_LOSS_REL, TOL_LSE_ABS, both_oracles, oracle_inputs,
                               rel_l2, run_fused, to_device)

pytestmark = pytest.mark.gpu


def _check(x, out, grad=1.0, tol_scale=1.0):
    """The GPU result against each of the two fp64 oracles (plain C++ and numpy)."""
    h, W = oracle_inputs(x)
    for name, orc in both_oracles():
        ref = orc.forward(h, W, x["idx"], x["t"], x["mask"], x["T"])
        g = orc.backward(h, W, x["idx"], x["t"], x["mask"], x["T"], grad_loss=grad)
        if ref["n_valid"] > 0:
            assert abs(out["loss"] - ref["loss"]) <= TOL_LOSS_REL * abs(ref["loss"]), (name, out["loss"], ref["loss"])
        else:
            assert out["loss"] == 0.0, name
        assert np.abs(out["lse"] - ref["lse"]).max() <= TOL_LSE_ABS, name
        if ref["n_valid"] > 0:
            assert rel_l2(out["dh"], g["dh"]) <= TOL_GRAD_REL_L2 * tol_scale, (name, rel_l2(out["dh"], g["dh"]))
            assert rel_l2(out["dW"], g["dW"]) <= TOL_GRAD_REL_L2 * tol_scale, (name, rel_l2(out["dW"], g["dW"]))
        else:
            assert not out["dh"].any() and not out["dW"].any(), name


SHAPES = [
    # N, d, V, K, T, index, chunk
    (300, 136, 1000, 16, 1.5, "uniform", 128),      # 3 chunks, ragged rows; d not a multiple of 64
    (257, 64, 1001, 8, 1.0, "uniform", 0),           # V odd: dz row stride padded; one ragged row tile
    (640, 256, 4096, 100, 2.0, "zipf1.1", 256),      # many teacher hits in the first vocab tiles
    (130, 384, 2304, 32, 0.5, "half-student", 0),    # teacher overlaps the student's top-K
    (96, 200, 777, 5, 1.0, "uniform", 0),            # everything ragged, N below one tile
    (1000, 96, 2500, 20, 1.0, "uniform", 384),       # chunk not a multiple of the 256-row pair tile
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "N{}_d{}_V{}_K{}".format(*s[:4]))
def test_parity_small(shape):
    N, d, V, K, T, index, chunk = shape
    x = synth.make_inputs(N, d, V, K, T, 0.05, index, seed=1000 + N)
    out = run_fused(to_device(x), chunk=chunk)
    _check(x, out)


def test_parity_tiny_config():
    x = synth.config_inputs(0)
    out = run_fused(to_device(x))
    _check(x, out)


def test_upstream_gradient_scales_dz():
    x = synth.make_inputs(200, 128, 600, 12, 1.0, 0.05, "uniform", seed=77)
    out = run_fused(to_device(x), grad=-2.5)
    _check(x, out, grad=-2.5)


def test_k1_single_teacher_entry():
    x = synth.make_inputs(150, 64, 512, 1, 1.0, 0.05, "uniform", seed=78)
    _check(x, run_fused(to_device(x)))


def test_all_rows_masked():
    x = synth.make_inputs(64, 64, 300, 4, 1.0, 0.0, "uniform", seed=79, n_pad=64)
    out = run_fused(to_device(x))
    _check(x, out)


def test_no_mask_and_minus_inf_teacher_logits():
    x = synth.make_inputs(70, 64, 400, 6, 1.0, 0.0, "uniform", seed=80)
    x["mask"] = None
    x["t"][3, 2:] = -np.inf       # partial: p = 0 on those entries
    x["t"][5, :] = -np.inf        # whole row: not a valid token
    out = run_fused(to_device(x))
    _check(x, out)


def test_single_row():
    x = synth.make_inputs(1, 64, 256, 4, 1.0, 0.0, "uniform", seed=81)
    _check(x, run_fused(to_device(x)))


def test_loss_and_lse_bitwise_chunk_invariant():
    x = synth.make_inputs(1000, 128, 2000, 20, 1.0, 0.05, "uniform", seed=82)
    xd = to_device(x)
    outs = []
    for chunk in (128, 384, 1024, 0):
        loss, lse = api.forward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], xd["T"], chunk)
        outs.append((loss.item(), lse.cpu().numpy()))
    for loss, lse in outs[1:]:
        assert loss == outs[0][0]
        assert np.array_equal(lse, outs[0][1])


def test_backward_deterministic():
    x = synth.make_inputs(600, 128, 3000, 16, 1.0, 0.05, "uniform", seed=83)
    xd = to_device(x)
    a = run_fused(xd, chunk=256)
    b = run_fused(xd, chunk=256)
    assert np.array_equal(a["dh"], b["dh"]) and np.array_equal(a["dW"], b["dW"])


def test_out_of_range_teacher_index_sets_status():
    x = synth.make_inputs(64, 64, 300, 4, 1.0, 0.0, "uniform", seed=84)
    x["idx"][10, 1] = 300  # == V
    xd = to_device(x)
    ws = api.alloc_workspace(64, 64, 300, 4)
    api.forward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], 1.0, ws=ws)
    assert api.get_status(ws) == 3
    x["idx"][10, 1] = 0 if 0 not in x["idx"][10] else 299
    xd = to_device(x)
    api.forward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], 1.0, ws=ws)
    assert api.get_status(ws) == 0


def test_autograd_loss_matches_oracle():
    x = synth.make_inputs(256, 128, 1024, 16, 2.0, 0.05, "uniform", seed=85)
    xd = to_device(x)
    h = xd["h"].clone().requires_grad_(True)
    W = xd["W"].clone().requires_grad_(True)
    loss = api.fkl_loss(h, W, xd["idx"], xd["t"], xd["mask"], 2.0)
    (3.0 * loss).backward()
    out = dict(loss=loss.item(), lse=None)
    hh, WW = oracle_inputs(x)
    ref = oracle.forward(hh, WW, x["idx"], x["t"], x["mask"], 2.0)
    g = oracle.backward(hh, WW, x["idx"], x["t"], x["mask"], 2.0, grad_loss=3.0)
    assert abs(out["loss"] - ref["loss"]) <= TOL_LOSS_REL * abs(ref["loss"])
    assert rel_l2(h.grad.double().cpu().numpy(), g["dh"]) <= TOL_GRAD_REL_L2
    assert rel_l2(W.grad.double().cpu().numpy(), g["dW"]) <= TOL_GRAD_REL_L2
    assert torch.isfinite(h.grad).all()


def test_row_shards_combine_to_full_batch():
    """The data-parallel reading of the loss, run shard after shard on one GPU.

    Rows split into R shards; shard r runs on its own with the upstream gradient
    g_r = N_valid_r / N_valid, so that its dz carries the global 1/N_valid.  Then
    loss = sum_r loss_r N_valid_r / N_valid, dh is the shards' dh stacked and
    dW = sum_r dW_r -- the only exchange a row-sharded job needs (the global
    N_valid before the step, one sum of loss and dW after it)."""
    x = synth.make_inputs(1100, 192, 3000, 24, 1.0, 0.05, "uniform", seed=90)
    full = run_fused(to_device(x), chunk=256)
    valid = oracle.row_valid(x["mask"], x["t"], x["T"])
    n_valid = int(valid.sum())
    bounds = [0, 300, 700, 1100]
    loss, dW, dh, lse = 0.0, 0.0, [], []
    for r0, r1 in zip(bounds[:-1], bounds[1:]):
        xs = dict(x, h=x["h"][r0:r1], idx=x["idx"][r0:r1], t=x["t"][r0:r1], mask=x["mask"][r0:r1])
        nv_r = int(valid[r0:r1].sum())
        out = run_fused(to_device(xs), chunk=256, grad=nv_r / n_valid)
        loss += out["loss"] * nv_r / n_valid
        dW = dW + out["dW"]
        dh.append(out["dh"])
        lse.append(out["lse"])
    # per-row work does not depend on which rows share a launch
    assert np.array_equal(np.concatenate(lse), full["lse"])
    assert abs(loss - full["loss"]) <= 1e-5 * abs(full["loss"])
    assert rel_l2(np.concatenate(dh), full["dh"]) <= 1e-3
    assert rel_l2(dW, full["dW"]) <= 1e-4
    _check(x, dict(loss=loss, lse=np.concatenate(lse), dh=np.concatenate(dh), dW=dW))


EDGE = [
    # N, d, V, K, T, index, chunk: the smallest hidden size, one partial vocabulary tile,
    # K = V, the largest K, extreme temperatures
    (200, 8, 777, 5, 1.0, "uniform", 0),
    (150, 64, 8, 3, 1.0, "uniform", 0),
    (130, 64, 40, 40, 1.0, "uniform", 0),
    (260, 96, 3000, 256, 1.0, "uniform", 128),
    (300, 128, 2000, 20, 0.05, "uniform", 128),
    (300, 128, 2000, 20, 20.0, "half-student", 0),
    (300, 4096, 1500, 16, 1.0, "uniform", 256),  # a wide hidden size: 8 wide dh / dW column tiles
    (256, 65536, 512, 8, 1.0, "uniform", 0),     # the largest hidden size the library takes
]


@pytest.mark.parametrize("shape", EDGE, ids=lambda s: "N{}_d{}_V{}_K{}_T{}".format(*s[:5]))
def test_edge_sizes(shape):
    N, d, V, K, T, index, chunk = shape
    x = synth.make_inputs(N, d, V, K, T, 0.05, index, seed=9200 + N + V)
    _check(x, run_fused(to_device(x), chunk=chunk))


def test_dW_rows_sum_to_zero():
    """sum_v dz_iv = T (sum_v q_iv - sum_k p_ik) / N_valid = 0 for every row, so the rows of
    dW sum to the zero vector -- up to the bf16 rounding of dz."""
    x = synth.make_inputs(700, 96, 3000, 24, 1.5, 0.05, "zipf1.1", seed=9400)
    out = run_fused(to_device(x), chunk=256)
    col = out["dW"].sum(axis=0)
    scale = np.abs(out["dW"]).sum(axis=0)
    assert np.all(np.abs(col) <= 2e-3 * scale), float((np.abs(col) / scale).max())


def test_uniform_student_closed_form():
    """W = 0: every logit is 0, so lse = log V / T * T = log V and KL_i = log V - H(p_i)."""
    x = synth.make_inputs(300, 64, 5000, 16, 2.0, 0.05, "uniform", seed=9401)
    x["W"] = np.zeros_like(x["W"])
    out = run_fused(to_device(x))
    assert np.abs(out["lse"] - np.log(5000.0)).max() <= 1e-5
    p = scipy_softmax(x["t"].astype(np.float64) / 2.0)
    H = -(p * np.log(p)).sum(axis=1)
    keep = x["mask"] != 0
    ref = 4.0 * (np.log(5000.0) - H[keep]).mean()
    assert abs(out["loss"] - ref) <= 1e-4 * abs(ref)


def scipy_softmax(a):
    import scipy.special
    return scipy.special.softmax(a, axis=1)
