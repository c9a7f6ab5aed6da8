"""Parity at the full workload sizes, in the launch configuration bench.py times.

The oracle's full fp64 forward (loss and lse of every row) is stored under
tests/golden/ by tests/golden/make_golden.py; here the GPU's loss and every lse
are compared with it, dh on 512 seeded sampled rows (plus the first and last) and
dW on ~500 sampled vocabulary rows (the most frequent teacher ids, random ids and
the ragged last tile) are recomputed by the oracle one by one.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from lm_head_kl_fkl_b300 import api, synth
from tests.gpu_helpers import TOL_GRAD_REL_L2, TOL_LOSS_REL, TOL_LSE_ABS, rel_l2, to_device

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(i):
    path = os.path.join(GOLDEN, f"oracle_forward_cfg{i}.npz")
    assert os.path.exists(path), f"missing {path}: run tests/golden/make_golden.py {i}"
    return np.load(path)


def _sample_vocab_rows(x, n_rand=384, n_hit=96, n_tail=32, seed=5):
    V = x["V"]
    rng = np.random.default_rng(seed)
    ids, counts = np.unique(x["idx"], return_counts=True)
    hit = ids[np.argsort(-counts, kind="stable")[:n_hit]]
    tail = np.arange(max(0, V - n_tail), V)
    rand = rng.choice(V, n_rand, replace=False)
    return np.unique(np.concatenate([hit, tail, rand]))


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_full_size_against_oracle(cfg):
    g = _golden(cfg)
    x = synth.config_inputs(cfg)
    assert str(g["fingerprint"]) == synth.fingerprint(x), "input generator drifted from the golden file"
    xd = to_device(x)
    loss, lse = api.forward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], x["T"])
    dh, dW = api.backward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], x["T"], lse)
    torch.cuda.synchronize()
    loss = float(loss.item())
    lse = lse.cpu().numpy().astype(np.float64)
    assert abs(loss - float(g["loss"])) <= TOL_LOSS_REL * abs(float(g["loss"])), (loss, float(g["loss"]))
    assert np.abs(lse - g["lse"]).max() <= TOL_LSE_ABS, np.abs(lse - g["lse"]).max()

    rng = np.random.default_rng(100 + cfg)
    rows = np.sort(rng.choice(x["N"], 512, replace=False))
    rows = np.unique(np.concatenate([rows, [0, x["N"] - 1]]))
    Wf = synth.bf16_bits_to_f64(x["W"])
    ref = oracle.rows_forward_backward(synth.bf16_bits_to_f64(x["h"][rows]), Wf, x["idx"][rows],
                                       x["t"][rows], x["mask"][rows], x["T"], np.arange(len(rows)))
    # rows_forward_backward counts N_valid inside the sample; rescale to the full job's N_valid
    n_valid = int(g["n_valid"])
    dh_ref = ref["dh"] * (ref["n_valid"] / n_valid)
    dh_gpu = dh[torch.from_numpy(rows).to(dh.device)].float().cpu().numpy()
    assert rel_l2(dh_gpu, dh_ref) <= TOL_GRAD_REL_L2, rel_l2(dh_gpu, dh_ref)

    vr = _sample_vocab_rows(x)
    hf = synth.bf16_bits_to_f64(x["h"])
    dW_ref = oracle.dW_rows(hf, Wf, x["idx"], x["t"], x["mask"], x["T"], g["lse"], vr)
    dW_gpu = dW[torch.from_numpy(vr).to(dW.device)].cpu().numpy().astype(np.float64)
    assert rel_l2(dW_gpu, dW_ref) <= TOL_GRAD_REL_L2, rel_l2(dW_gpu, dW_ref)


def test_chunk_sweep_loss_agrees():
    """Llama-like head: the loss is identical across chunk sizes 512, 1024 and 2048."""
    g = _golden(2)
    x = synth.config_inputs(2)
    xd = to_device(x)
    losses = []
    for chunk in (512, 1024, 2048):
        loss, lse = api.forward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], x["T"], chunk)
        losses.append(float(loss.item()))
    assert losses[0] == losses[1] == losses[2], losses
    assert abs(losses[0] - float(g["loss"])) <= TOL_LOSS_REL * abs(float(g["loss"]))
