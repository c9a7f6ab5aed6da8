"""The loss's calls enqueue only on the caller's stream, with no host synchronisation
and no allocation, so a whole training-step loss can be captured in a CUDA graph and
replayed: the replays give the eager results bit for bit."""
import numpy as np
import pytest
import torch

from lm_head_kl_fkl_b300 import api, synth
from tests.gpu_helpers import to_device

pytestmark = pytest.mark.gpu


def test_forward_backward_replay_in_a_cuda_graph():
    x = synth.make_inputs(700, 136, 3001, 24, 1.5, 0.05, "uniform", seed=9100)
    xd = to_device(x)
    N, d, V, K = 700, 136, 3001, 24
    dev = xd["h"].device
    ws = api.alloc_workspace(N, d, V, K, 256, dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    dh = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    dW = torch.empty((V, d), dtype=torch.float32, device=dev)

    def step():
        api.forward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], xd["T"], 256, ws=ws, loss=loss, lse=lse)
        api.backward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], xd["T"], lse, chunk=256, ws=ws, dh=dh, dW=dW)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # eager warm-up: first-use set-up happens outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    ref = (loss.clone(), lse.clone(), dh.clone(), dW.clone())

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        loss.zero_(), lse.zero_(), dh.zero_(), dW.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert api.get_status(ws) == 0
        for a, b in zip((loss, lse, dh, dW), ref):
            assert torch.equal(a, b)


def test_one_call_path_replays_in_a_cuda_graph():
    x = synth.make_inputs(500, 128, 2500, 16, 1.0, 0.05, "uniform", seed=9101)
    xd = to_device(x)
    dev = xd["h"].device
    ws = api.alloc_workspace(500, 128, 2500, 16, 128, dev)
    out = dict(loss=torch.empty(1, device=dev), lse=torch.empty(500, device=dev),
               dh=torch.empty((500, 128), dtype=torch.bfloat16, device=dev),
               dW=torch.empty((2500, 128), dtype=torch.float32, device=dev))

    def step():
        api.forward_backward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], xd["T"], chunk=128, ws=ws, **out)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    ref = {k: v.clone() for k, v in out.items()}
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for v in out.values():
        v.zero_()
    g.replay()
    torch.cuda.synchronize()
    for k in out:
        assert torch.equal(out[k], ref[k]), k
