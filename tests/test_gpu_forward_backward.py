"""fkl_forward_backward (loss and gradients in one call, logits kept per chunk
instead of recomputed) against the fp64 oracle, and against the two-call path."""
import numpy as np
import pytest
import torch

import oracle
from lm_head_kl_fkl_b300 import api, synth
from tests.gpu_helpers import (TOL_GRAD_REL_L2, TOL_LOSS_REL, TOL_LSE_ABS, oracle_inputs, rel_l2,
                               run_fused, to_device)
from tests.test_gpu_parity import SHAPES, _check

pytestmark = pytest.mark.gpu


def run_one_call(xd, chunk=0, grad=None):
    g = None if grad is None else torch.tensor([grad], dtype=torch.float32, device=xd["h"].device)
    loss, lse, dh, dW = api.forward_backward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], xd["T"],
                                             grad_loss=g, chunk=chunk)
    torch.cuda.synchronize()
    return dict(loss=float(loss.item()), lse=lse.cpu().numpy().astype(np.float64),
                dh=dh.float().cpu().numpy().astype(np.float64), dW=dW.cpu().numpy().astype(np.float64))


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "N{}_d{}_V{}_K{}".format(*s[:4]))
def test_parity_small(shape):
    N, d, V, K, T, index, chunk = shape
    x = synth.make_inputs(N, d, V, K, T, 0.05, index, seed=1000 + N)
    xd = to_device(x)
    one = run_one_call(xd, chunk=chunk)
    _check(x, one)
    two = run_fused(xd, chunk=chunk)
    # same loss pass up to the order of the per-tile max / sum; dz from fp16-kept logits
    assert abs(one["loss"] - two["loss"]) <= 1e-5 * abs(two["loss"])
    assert np.abs(one["lse"] - two["lse"]).max() <= 1e-5
    assert rel_l2(one["dh"], two["dh"]) <= 5e-3
    assert rel_l2(one["dW"], two["dW"]) <= 5e-3


def test_tiny_config_and_upstream_gradient():
    x = synth.config_inputs(0)
    _check(x, run_one_call(to_device(x), grad=-1.75), grad=-1.75)


def test_degenerate_rows():
    x = synth.make_inputs(70, 64, 400, 6, 1.0, 0.0, "uniform", seed=80)
    x["mask"] = None
    x["t"][3, 2:] = -np.inf
    x["t"][5, :] = -np.inf
    _check(x, run_one_call(to_device(x)))
    y = synth.make_inputs(64, 64, 300, 4, 1.0, 0.0, "uniform", seed=79, n_pad=64)
    _check(y, run_one_call(to_device(y)))
    z = synth.make_inputs(150, 64, 512, 1, 1.0, 0.05, "uniform", seed=78)
    _check(z, run_one_call(to_device(z)))


def test_repeated_teacher_ids_are_summed():
    # outside the precondition, but defined: s sums p over repeated ids, as in the two-call path
    x = synth.make_inputs(40, 64, 256, 6, 1.0, 0.0, "uniform", seed=91)
    x["idx"][4, 1] = x["idx"][4, 0]
    x["idx"][9, 5] = x["idx"][9, 2]
    xd = to_device(x)
    one, two = run_one_call(xd), run_fused(xd)
    assert rel_l2(one["dh"], two["dh"]) <= 5e-3 and rel_l2(one["dW"], two["dW"]) <= 5e-3
    h, W = oracle_inputs(x)
    g = oracle.backward(h, W, x["idx"], x["t"], x["mask"], x["T"])
    assert rel_l2(one["dW"], g["dW"]) <= TOL_GRAD_REL_L2


def test_bad_teacher_id_sets_status():
    x = synth.make_inputs(64, 64, 300, 4, 1.0, 0.0, "uniform", seed=84)
    x["idx"][10, 1] = 300
    xd = to_device(x)
    ws = api.alloc_workspace(64, 64, 300, 4)
    api.forward_backward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], 1.0, ws=ws)
    assert api.get_status(ws) == 3


def test_full_size_bench_workload():
    """The gpt-oss-20b-like workload at full size: loss and every lse against the
    stored oracle values, dh and dW on sampled rows against the oracle."""
    from tests.test_gpu_full_size import _golden, _sample_vocab_rows
    g = _golden(3)
    x = synth.config_inputs(3)
    xd = to_device(x)
    loss, lse, dh, dW = api.forward_backward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], x["T"])
    torch.cuda.synchronize()
    assert abs(float(loss.item()) - float(g["loss"])) <= TOL_LOSS_REL * abs(float(g["loss"]))
    assert np.abs(lse.cpu().numpy().astype(np.float64) - g["lse"]).max() <= TOL_LSE_ABS
    rng = np.random.default_rng(103)
    rows = np.unique(np.concatenate([np.sort(rng.choice(x["N"], 192, replace=False)), [0, x["N"] - 1]]))
    Wf = synth.bf16_bits_to_f64(x["W"])
    ref = oracle.rows_forward_backward(synth.bf16_bits_to_f64(x["h"][rows]), Wf, x["idx"][rows],
                                       x["t"][rows], x["mask"][rows], x["T"], np.arange(len(rows)))
    dh_ref = ref["dh"] * (ref["n_valid"] / int(g["n_valid"]))
    dh_gpu = dh[torch.from_numpy(rows).to(dh.device)].float().cpu().numpy()
    assert rel_l2(dh_gpu, dh_ref) <= TOL_GRAD_REL_L2
    vr = _sample_vocab_rows(x)
    dW_ref = oracle.dW_rows(synth.bf16_bits_to_f64(x["h"]), Wf, x["idx"], x["t"], x["mask"], x["T"], g["lse"], vr)
    dW_gpu = dW[torch.from_numpy(vr).to(dW.device)].cpu().numpy().astype(np.float64)
    assert rel_l2(dW_gpu, dW_ref) <= TOL_GRAD_REL_L2


def test_autograd_keep_logits_matches_oracle_and_recompute():
    x = synth.make_inputs(256, 128, 1024, 16, 2.0, 0.05, "uniform", seed=85)
    xd = to_device(x)
    grads = {}
    for keep in (False, True):
        h = xd["h"].clone().requires_grad_(True)
        W = xd["W"].clone().requires_grad_(True)
        loss = api.fkl_loss(h, W, xd["idx"], xd["t"], xd["mask"], 2.0, keep_logits=keep)
        (3.0 * loss).backward()
        grads[keep] = (loss.item(), h.grad.double().cpu().numpy(), W.grad.double().cpu().numpy())
    hh, WW = oracle_inputs(x)
    ref = oracle.forward(hh, WW, x["idx"], x["t"], x["mask"], 2.0)
    g = oracle.backward(hh, WW, x["idx"], x["t"], x["mask"], 2.0, grad_loss=3.0)
    loss, dh, dW = grads[True]
    assert abs(loss - ref["loss"]) <= TOL_LOSS_REL * abs(ref["loss"])
    assert rel_l2(dh, g["dh"]) <= TOL_GRAD_REL_L2 and rel_l2(dW, g["dW"]) <= TOL_GRAD_REL_L2
    assert rel_l2(dh, grads[False][1]) <= 5e-3 and rel_l2(dW, grads[False][2]) <= 5e-3


def test_scale_grads_by_one_is_exact():
    x = synth.make_inputs(200, 64, 700, 8, 1.0, 0.05, "uniform", seed=86)
    xd = to_device(x)
    _, _, dh, dW = api.forward_backward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], 1.0)
    a, b = dh.clone(), dW.clone()
    import ctypes
    from lm_head_kl_fkl_b300 import _lib
    one = torch.ones(1, dtype=torch.float32, device=dh.device)
    st = _lib.lib().fkl_scale_grads(ctypes.c_void_p(dh.data_ptr()), ctypes.c_void_p(dW.data_ptr()), 200, 64, 700,
                                    ctypes.c_void_p(one.data_ptr()),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert st == 0 and torch.equal(a, dh) and torch.equal(b, dW)
