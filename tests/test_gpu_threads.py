"""The library called from two host threads at once, each on its own stream and
workspace, with the profiling hooks on: results bitwise equal to the same calls
made one after the other, and every launch of both threads recorded."""
import threading

import numpy as np
import pytest
import torch

from lm_head_kl_fkl_b300 import api, synth
from tests.gpu_helpers import to_device

pytestmark = pytest.mark.gpu

SHAPES = [(640, 256, 8192 + 72, 16, 1.0), (384, 192, 5000, 24, 2.0)]


def _step(xd, ws):
    loss, lse = api.forward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], xd["T"], 256, ws=ws)
    dh, dW = api.backward(xd["h"], xd["W"], xd["idx"], xd["t"], xd["mask"], xd["T"], lse, chunk=256, ws=ws)
    return loss, lse, dh, dW


def _host(r):
    return [t.float().cpu().numpy() for t in r]


def test_two_threads_two_streams():
    xds = [to_device(synth.make_inputs(N, d, V, K, T, 0.05, "uniform", seed=4100 + i))
           for i, (N, d, V, K, T) in enumerate(SHAPES)]
    wss = [api.alloc_workspace(xd["h"].shape[0], xd["h"].shape[1], xd["W"].shape[0], xd["idx"].shape[1], 256)
           for xd in xds]
    alone = [_host(_step(xd, ws)) for xd, ws in zip(xds, wss)]
    torch.cuda.synchronize()
    launches_alone = api.launch_count()
    _step(xds[0], wss[0])
    torch.cuda.synchronize()
    per_step0 = api.launch_count() - launches_alone
    launches_alone = api.launch_count()
    _step(xds[1], wss[1])
    torch.cuda.synchronize()
    per_step1 = api.launch_count() - launches_alone

    reps = 4
    streams = [torch.cuda.Stream() for _ in xds]
    out = [None, None]
    errors = []
    start = threading.Barrier(2)

    def work(i):
        try:
            with torch.cuda.stream(streams[i]):
                start.wait()
                for _ in range(reps):
                    out[i] = _step(xds[i], wss[i])
                streams[i].synchronize()
        except Exception as e:  # reported on the main thread
            errors.append(e)

    api.profile_reset()
    api.profile_enable(True)
    try:
        threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
        for t in threads:
            t.start()
        for t in threads:
            t.join(timeout=120)
        assert not any(t.is_alive() for t in threads)
        torch.cuda.synchronize()
        prof = api.profile_read()
    finally:
        api.profile_enable(False)
        api.profile_reset()
    assert not errors, errors
    for i in range(2):
        for a, b in zip(alone[i], _host(out[i])):
            assert np.array_equal(a, b)
    recorded = sum(v[1] for v in prof.values())
    assert recorded == reps * (per_step0 + per_step1)
    assert all(v[0] > 0 for v in prof.values())
