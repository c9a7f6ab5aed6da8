"""The C ABI from a plain C program: tests/c_abi/fkl_c_demo.c is compiled with gcc
against include/fkl.h, libfkl.so and the CUDA runtime, runs the loss through
fkl_forward / fkl_backward / fkl_forward_noalloc, and its outputs are compared with
the fp64 oracle on the same inputs, rebuilt here from the program's counter hash."""
import os
import subprocess

import numpy as np
import pytest

import oracle
from lm_head_kl_fkl_b300 import _lib, synth
from tests.gpu_helpers import TOL_GRAD_REL_L2, TOL_LOSS_REL, TOL_LSE_ABS, rel_l2

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
N, D, V, K, T = 300, 128, 2048, 16, 1.5
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _mix32(x):
    x = x.astype(np.uint64)
    m = np.uint64(0xFFFFFFFF)
    x ^= x >> np.uint64(16)
    x = (x * np.uint64(0x7FEB352D)) & m
    x ^= x >> np.uint64(15)
    x = (x * np.uint64(0x846CA68B)) & m
    x ^= x >> np.uint64(16)
    return x


def _unif(i, s):
    i = np.asarray(i, dtype=np.uint64)
    key = ((i * np.uint64(2654435761)) & np.uint64(0xFFFFFFFF)) ^ np.uint64((s * 0x9E3779B9) & 0xFFFFFFFF)
    return (_mix32(key) >> np.uint64(8)).astype(np.float32) / np.float32(16777216.0)


def _inputs():
    h = synth.f32_to_bf16_bits((np.float32(2.0) * _unif(np.arange(N * D), 1) - np.float32(1.0)).reshape(N, D))
    W = synth.f32_to_bf16_bits((np.float32(0.2) * _unif(np.arange(V * D), 2) - np.float32(0.1)).reshape(V, D))
    r = np.arange(N, dtype=np.int64)[:, None]
    k = np.arange(K, dtype=np.int64)[None, :]
    idx = ((r * 131 + k * 997) % V).astype(np.int32)
    t = (np.float32(4.0) * _unif(np.arange(N * K), 3) - np.float32(2.0)).reshape(N, K)
    mask = (np.arange(N) % 17 != 0).astype(np.uint8)
    return h, W, idx, t, mask


def test_plain_c_program(tmp_path):
    exe = tmp_path / "fkl_c_demo"
    lib_dir = os.path.dirname(_lib.LIB_PATH)
    cmd = ["gcc", "-O2", "-std=c99", os.path.join(HERE, "c_abi", "fkl_c_demo.c"), "-o", str(exe),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", lib_dir, "-lfkl", f"-Wl,-rpath,{lib_dir}", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = tmp_path / "out.bin"
    r = subprocess.run([str(exe), str(out)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    raw = out.read_bytes()
    loss = np.frombuffer(raw, np.float32, 2, 0)
    lse = np.frombuffer(raw, np.float32, N, 8).astype(np.float64)
    dh = synth.bf16_bits_to_f64(np.frombuffer(raw, np.uint16, N * D, 8 + 4 * N).reshape(N, D))
    dW = np.frombuffer(raw, np.float32, V * D, 8 + 4 * N + 2 * N * D).reshape(V, D).astype(np.float64)
    assert loss[0] == loss[1]  # the no-alloc forward runs the same kernels

    h, W, idx, t, mask = _inputs()
    hf, Wf = synth.bf16_bits_to_f64(h), synth.bf16_bits_to_f64(W)
    ref = oracle.forward(hf, Wf, idx, t, mask, T)
    g = oracle.backward(hf, Wf, idx, t, mask, T)
    assert abs(float(loss[0]) - ref["loss"]) <= TOL_LOSS_REL * abs(ref["loss"])
    assert np.abs(lse - ref["lse"]).max() <= TOL_LSE_ABS
    assert rel_l2(dh, g["dh"]) <= TOL_GRAD_REL_L2
    assert rel_l2(dW, g["dW"]) <= TOL_GRAD_REL_L2
