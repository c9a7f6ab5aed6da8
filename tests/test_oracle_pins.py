"""Both fp64 oracles (numpy and plain C++) against their pins, and planted
mistakes against the pins.

A planted mistake is a textual edit of a copy of an oracle's source -- loaded as
a separate module (numpy) or compiled into a separate library (C++) on the CPU;
at least one pin must reject each mutant.  The two oracles are also compared with
each other on the tiny workload (they share no code).
"""
import importlib.util
import os
import types

import numpy as np
import pytest

import oracle
from oracle import cpp
from lm_head_kl_fkl_b300 import synth
from tests import oracle_pins as P

ORACLE_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")
ORACLE_SRC = os.path.join(ORACLE_DIR, "fkl_oracle.py")


@pytest.fixture(scope="module")
def cpp_oracle():
    return cpp.load()


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle)


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin_cpp(pin, cpp_oracle):
    pin(cpp_oracle)


def test_numpy_and_cpp_oracles_agree_on_tiny_workload(cpp_oracle):
    x = synth.config_inputs(0)
    h, W = synth.bf16_bits_to_f64(x["h"]), synth.bf16_bits_to_f64(x["W"])
    a = oracle.forward(h, W, x["idx"], x["t"], x["mask"], x["T"])
    b = cpp_oracle.forward(h, W, x["idx"], x["t"], x["mask"], x["T"])
    assert a["n_valid"] == b["n_valid"]
    assert abs(a["loss"] - b["loss"]) <= 1e-12 * abs(a["loss"])
    np.testing.assert_allclose(a["lse"], b["lse"], rtol=1e-13)
    ga = oracle.backward(h, W, x["idx"], x["t"], x["mask"], x["T"])
    gb = cpp_oracle.backward(h, W, x["idx"], x["t"], x["mask"], x["T"])
    np.testing.assert_allclose(ga["dh"], gb["dh"], rtol=1e-9, atol=1e-15)
    np.testing.assert_allclose(ga["dW"], gb["dW"], rtol=1e-9, atol=1e-15)


def _mutant(old, new):
    with open(ORACLE_SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


MUTATIONS = {
    "drop_T_squared": ("float(T) ** 2 * kl[valid]", "kl[valid]"),
    "teacher_ignores_T": ("u = np.asarray(tlogit, dtype=np.float64) / float(T)",
                          "u = np.asarray(tlogit, dtype=np.float64)"),
    "student_normaliser_over_K_only": (
        "    a = z / float(T)\n    lse = _logsumexp_rows(a)\n    a_idx",
        "    a = z / float(T)\n    lse = _logsumexp_rows(np.take_along_axis(a, idx.astype(np.int64), axis=1))\n    a_idx"),
    "gradient_sign": ("return coef[:, None] * (q - s), lse", "return coef[:, None] * (s - q), lse"),
    "gradient_drops_teacher": ("return coef[:, None] * (q - s), lse", "return coef[:, None] * q, lse"),
    "index_off_by_one": ("a_idx = np.take_along_axis(a, idx.astype(np.int64), axis=1)",
                         "a_idx = np.take_along_axis(a, (idx.astype(np.int64) + 1) % a.shape[1], axis=1)"),
    "mean_over_all_rows": ("kl[valid].sum() / n_valid", "kl[valid].sum() / N"),
    "reverse_kl": ("kl = np.where(p > 0, p * (logp - logq), 0.0).sum(axis=1)",
                   "kl = np.where(p > 0, np.exp(logq) * (logq - logp), 0.0).sum(axis=1)"),
    "dW_transposed_operand": ("coef[r0:r1])\n        dh[r0:r1] = dz @ W\n        dW += dz.T @ h[r0:r1]",
                              "coef[r0:r1])\n        dh[r0:r1] = dz @ W\n        dW += (dz.T @ h[r0:r1])[::-1]"),
    "lse_missing_max_shift": ("return m + np.log(np.exp(a - m[:, None]).sum(axis=1))",
                              "return np.log(np.exp(a - m[:, None]).sum(axis=1))"),
    "mixture_ce_without_lse": ("ce[r0:r1] = lse1[r0:r1] - z[np.arange(r1 - r0), label[r0:r1]]",
                               "ce[r0:r1] = - z[np.arange(r1 - r0), label[r0:r1]]"),
    "mixture_weights_swapped": ("(1.0 - float(alpha)) * ce_mean", "float(alpha) * ce_mean"),
    "mixture_grad_label_sign": ("q1[np.arange(r1 - r0), label[r0:r1]] -= 1.0",
                                "q1[np.arange(r1 - r0), label[r0:r1]] += 1.0"),
    "topk_ascending": ('order = np.argsort(-z, axis=1, kind="stable")[:, :K]',
                       'order = np.argsort(z, axis=1, kind="stable")[:, :K]'),
    "topk_ties_to_larger_id": ('order = np.argsort(-z, axis=1, kind="stable")[:, :K]',
                               'order = (z.shape[1] - 1 - np.argsort(-z[:, ::-1], axis=1, kind="stable"))[:, :K]'),
}

# The same kinds of mistake, planted in the C++ oracle's source.
CPP_MUTATIONS = {
    "drop_T_squared": ("*loss = nv > 0 ? T * T * sum", "*loss = nv > 0 ? sum"),
    "teacher_ignores_T": ("bool teacher_row(const double* t, int64_t K, double T, double* p) {",
                          "bool teacher_row(const double* t, int64_t K, double T_, double* p) {\n"
                          "    const double T = 1.0;\n    (void)T_;"),
    "student_normaliser_truncated": ("*lse = lse_row(z, V, T);", "*lse = lse_row(z, K, T);"),
    "gradient_sign": ("dz[v] *= coef;", "dz[v] *= -coef;"),
    "gradient_drops_teacher": ("for (int64_t k = 0; k < K; ++k) dz[idx[k]] -= p[k];", ""),
    "index_off_by_one": ("const double logq = z[idx[k]] / T - lse;",
                         "const double logq = z[idx[k] == 0 ? 1 : idx[k] - 1] / T - lse;"),
    "mean_over_all_rows": ("T * T * sum / static_cast<double>(nv)", "T * T * sum / static_cast<double>(N)"),
    "reverse_kl": ("kl += p[k] * (std::log(p[k]) - logq);", "kl += std::exp(logq) * (logq - std::log(p[k]));"),
    "dW_rows_permuted": ("double* dwv = dW + v * d;\n                for (int64_t i = r0; i < r1; ++i) {",
                         "double* dwv = dW + (V - 1 - v) * d;\n                for (int64_t i = r0; i < r1; ++i) {"),
    "lse_missing_max_shift": ("return m + std::log(s);", "return std::log(s);"),
    "dh_wrong_weight_row": ("dhi[j] += dzr[v] * W[v * d + j];", "dhi[j] += dzr[v] * W[((v + 1) % V) * d + j];"),
    "mixture_ce_without_lse": ("ce[i] = lse1[i] - z[label[i]];", "ce[i] = -z[label[i]];"),
    "mixture_grad_label_sign": ("q1[label[i]] -= 1.0;", "q1[label[i]] += 1.0;"),
    "topk_ascending": ("return z[a] > z[c] || (z[a] == z[c] && a < c);",
                       "return z[a] < z[c] || (z[a] == z[c] && a < c);"),
    "topk_ties_to_larger_id": ("return z[a] > z[c] || (z[a] == z[c] && a < c);",
                               "return z[a] > z[c] || (z[a] == z[c] && a > c);"),
}


def _rejected_by(mod):
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(mod)
        except Exception:  # AssertionError or a shape error both reject the mutant
            caught.append(pin.__name__)
    return caught


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    assert _rejected_by(_mutant(*MUTATIONS[name])), f"no pin rejects the planted mistake {name}"


@pytest.mark.parametrize("name", sorted(CPP_MUTATIONS))
def test_planted_mistake_is_caught_cpp(name, tmp_path):
    old, new = CPP_MUTATIONS[name]
    with open(cpp.SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    mutant_src = tmp_path / "mutant.cpp"
    mutant_src.write_text(src.replace(old, new))
    lib = cpp.compile_library(str(mutant_src), str(tmp_path / "libmutant.so"))
    assert _rejected_by(cpp.CppOracle(lib)), f"no pin rejects the planted mistake {name}"
