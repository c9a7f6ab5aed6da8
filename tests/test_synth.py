"""The seeded input generator: determinism and the structure each workload promises."""
import numpy as np
import pytest

from lm_head_kl_fkl_b300 import synth


def test_bf16_rounding_is_rne():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e-39, 65504.0], dtype=np.float32)
    b = synth.f32_to_bf16_bits(x)
    back = synth.bf16_bits_to_f32(b)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: ties go to the even mantissa (1.0)
    assert back[1] == np.float32(1.0)
    # 1 + 3*2^-8 is a tie between 1+2^-7 and 1+2^-6: even is 1 + 2^-6
    assert back[2] == np.float32(1.015625)
    assert back[0] == 1.0 and back[3] == -2.5
    rng = np.random.default_rng(0)
    y = rng.standard_normal(10000).astype(np.float32)
    yb = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(y))
    assert np.all(np.abs(yb - y) <= np.abs(y) * 2.0 ** -8)


def test_deterministic_and_distinct():
    a = synth.make_inputs(300, 64, 1000, 20, 1.0, 0.05, "uniform", seed=5)
    b = synth.make_inputs(300, 64, 1000, 20, 1.0, 0.05, "uniform", seed=5)
    for k in ("h", "W", "idx", "t", "mask"):
        assert np.array_equal(a[k], b[k])
    assert synth.fingerprint(a) == synth.fingerprint(b)
    s = np.sort(a["idx"], axis=1)
    assert np.all(s[:, 1:] != s[:, :-1])
    assert a["idx"].min() >= 0 and a["idx"].max() < 1000
    assert np.all(np.diff(a["t"], axis=1) <= 0)
    assert int((a["mask"] == 0).sum()) == 15


def test_zipf_skew():
    x = synth.make_inputs(200, 16, 5000, 30, 1.0, 0.02, "zipf1.1", seed=9)
    s = np.sort(x["idx"], axis=1)
    assert np.all(s[:, 1:] != s[:, :-1])
    # low ids dominate: id 0 appears in most rows, the top half of the vocab rarely
    assert (x["idx"] == 0).any(axis=1).mean() > 0.9
    assert (x["idx"] >= 2500).mean() < 0.2


def test_half_student_overlap():
    x = synth.make_inputs(64, 32, 512, 16, 2.0, 0.05, "half-student", seed=3)
    h = synth.bf16_bits_to_f64(x["h"])
    W = synth.bf16_bits_to_f64(x["W"])
    top = np.argsort(-(h @ W.T), axis=1)[:, :16]
    overlap = np.array([len(set(top[i]) & set(x["idx"][i])) for i in range(64)])
    assert (overlap >= 10).sum() == 32  # exactly the student half keeps most of its top-K
    s = np.sort(x["idx"], axis=1)
    assert np.all(s[:, 1:] != s[:, :-1])


@pytest.mark.parametrize("i", [0])
def test_config_shapes(i):
    x = synth.config_inputs(i)
    c = synth.CONFIGS[i]
    assert x["h"].shape == (c.N, c.d) and x["W"].shape == (c.V, c.d)
    assert x["idx"].shape == (c.N, c.K) and x["t"].dtype == np.float32
    w = synth.bf16_bits_to_f64(x["W"])
    assert abs(w.std() * np.sqrt(c.d) - 1.0) < 0.02
