"""The fp64 oracle against its pins, and planted mistakes against the pins.

A planted mistake is a textual edit of a copy of the oracle's source, loaded as a
separate module on the CPU; at least one pin must reject each mutant.
"""
import importlib.util
import os
import types

import pytest

import oracle
from tests import oracle_pins as P

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "oracle", "fkl_oracle.py")


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle)


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
    "dW_transposed_operand": ("dW += dz.T @ h[r0:r1]", "dW += (dz.T @ h[r0:r1])[::-1]"),
    "lse_missing_max_shift": ("return m + np.log(np.exp(a - m[:, None]).sum(axis=1))",
                              "return np.log(np.exp(a - m[:, None]).sum(axis=1))"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    mod = _mutant(*MUTATIONS[name])
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(mod)
        except Exception:  # AssertionError or a shape error both reject the mutant
            caught.append(pin.__name__)
    assert caught, f"no pin rejects the planted mistake {name}"
