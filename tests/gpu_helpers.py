"""Helpers shared by the GPU tests: device copies of generator output, one fused
forward + backward through the library, and the error measures of the spec."""
import numpy as np
import torch

from lm_head_kl_fkl_b300 import api, synth

# Parity bar: |dloss|/|loss| <= 1e-3, |dlse| <= 1e-3 absolute, rel. L2 of dh, dW <= 2e-2.
TOL_LOSS_REL = 1e-3
TOL_LSE_ABS = 1e-3
TOL_GRAD_REL_L2 = 2e-2


def to_device(x, device="cuda"):
    return dict(
        h=torch.from_numpy(x["h"].view(np.int16)).view(torch.bfloat16).to(device),
        W=torch.from_numpy(x["W"].view(np.int16)).view(torch.bfloat16).to(device),
        idx=torch.from_numpy(x["idx"]).to(device),
        t=torch.from_numpy(x["t"]).to(device),
        mask=None if x["mask"] is None else torch.from_numpy(x["mask"]).to(device),
        T=x["T"],
    )


def run_fused(xd, chunk=0, grad=None):
    loss, lse = api.forward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], xd["T"], chunk)
    g = None if grad is None else torch.tensor([grad], dtype=torch.float32, device=xd["h"].device)
    dh, dW = api.backward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], xd["T"], lse,
                          grad_loss=g, chunk=chunk)
    torch.cuda.synchronize()
    return dict(loss=float(loss.item()), lse=lse.cpu().numpy().astype(np.float64),
                dh=dh.float().cpu().numpy().astype(np.float64), dW=dW.cpu().numpy().astype(np.float64))


def rel_l2(a, b):
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def oracle_inputs(x):
    return synth.bf16_bits_to_f64(x["h"]), synth.bf16_bits_to_f64(x["W"])


def both_oracles():
    """[(name, oracle)] for the two independent fp64 oracles: the plain C++ one (one
    full logit row at a time, loops only) and the numpy one (a library matmul)."""
    import oracle
    from oracle import cpp
    return [("cpp", cpp.load()), ("numpy", oracle)]
