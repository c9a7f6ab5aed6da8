"""Seeded synthetic inputs for the fused top-K forward-KL loss.

This module only *draws* inputs: student hidden states h, the LM-head weight W,
the offline teacher cache (top-K indices and logits) and the padding mask.  It
holds none of the loss arithmetic, and both the CPU oracle (via the tests) and
the CUDA path consume exactly the arrays it returns.

Workloads follow the five distillation shapes used across this project:

=====  ========  ======  =======  ===  ===  =====  ======================================
name   N         d       V        K    T    pad    teacher indices
=====  ========  ======  =======  ===  ===  =====  ======================================
tiny   256       256     4096     16   1    5 %    uniform distinct
small  4096      2048    32768    100  2    5 %    half uniform, half student top-100 +-10 %
llama  8192      3072    128256   100  1    5 %    uniform distinct
oss20  32768     2880    201088   100  1    2 %    Zipf(1.1) distinct
oss120 131072    2880    201088   100  1    2 %    uniform distinct
=====  ========  ======  =======  ===  ===  =====  ======================================

V = 201088 is the gpt-oss vocabulary and K = 100 the cached top-100 named by
"Effektivnaya distillyatsiya znaniy" (malakhovai.ru, paragraph 2 and 4) and
"Wissensdestillation mit deutlich weniger GPU-Speicher" (dailytechsnack.ch,
"Teacher-Ausgaben einmalig zwischenspeichern").

Recipe (seed s, one numpy PCG64 stream, draws in this order):
  1. h  = bf16_rne(N(0,1))           [N, d], float32 normals drawn in row blocks
  2. W  = bf16_rne(N(0,1) / sqrt(d)) [V, d]
  3. t  = sort_desc(3 * N(0,1))      [N, K] float32 teacher logits
  4. idx: K distinct ids per row; duplicates are re-drawn until a row is distinct
     (uniform ids: a uniformly random ordered K-subset, the same law as a
     partial Fisher-Yates shuffle; Zipf ids: P(v) ~ (v+1)^-1.1 by inverse CDF).
     For the "half-student" mode, a seeded half of the rows instead takes the
     student's own top-K ids (fp64 logits of the bf16 h and W), each replaced
     with probability 0.10 by a uniform id not already in the row.  Column k of
     idx pairs with column k of t, so the teacher's rank order follows the
     student's.
  5. mask: exactly round(pad * N) padding rows (mask 0) from a seeded permutation.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Optional

import numpy as np

BASE_SEED = 0x464B4C00


@dataclasses.dataclass(frozen=True)
class Shape:
    name: str
    N: int
    d: int
    V: int
    K: int
    T: float
    pad_frac: float
    index: str  # "uniform" | "zipf1.1" | "half-student"


CONFIGS = (
    Shape("tiny", 256, 256, 4096, 16, 1.0, 0.05, "uniform"),
    Shape("small-lm-head", 4096, 2048, 32768, 100, 2.0, 0.05, "half-student"),
    Shape("llama-8b-to-3b-head", 8192, 3072, 128256, 100, 1.0, 0.05, "uniform"),
    Shape("gpt-oss-20b-long-context", 32768, 2880, 201088, 100, 1.0, 0.02, "zipf1.1"),
    Shape("gpt-oss-120b-memory-stress", 131072, 2880, 201088, 100, 1.0, 0.02, "uniform"),
)


def config_seed(i: int) -> int:
    return BASE_SEED + i


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even); returns the bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """bf16 -> float64 is exact."""
    return bf16_bits_to_f32(b).astype(np.float64)


def _normals_bf16(rng: np.random.Generator, rows: int, cols: int, scale: float,
                  block: int = 4096) -> np.ndarray:
    out = np.empty((rows, cols), dtype=np.uint16)
    for r0 in range(0, rows, block):
        r1 = min(rows, r0 + block)
        x = rng.standard_normal((r1 - r0, cols), dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        out[r0:r1] = f32_to_bf16_bits(x)
    return out


def _make_distinct(idx: np.ndarray, redraw) -> np.ndarray:
    """Re-draw later duplicates in each row (in column order) until every row is distinct."""
    while True:
        order = np.argsort(idx, axis=1, kind="stable")
        s = np.take_along_axis(idx, order, axis=1)
        dup = np.zeros(s.shape, dtype=bool)
        dup[:, 1:] = s[:, 1:] == s[:, :-1]
        if not dup.any():
            return idx
        rr, cc = np.nonzero(dup)
        idx[rr, order[rr, cc]] = redraw(len(rr))


def _uniform_distinct(rng, N, K, V):
    if K > V:
        raise ValueError("K must not exceed V")
    idx = rng.integers(0, V, size=(N, K), dtype=np.int64)
    return _make_distinct(idx, lambda n: rng.integers(0, V, size=n, dtype=np.int64))


def zipf_cdf(V: int, a: float = 1.1) -> np.ndarray:
    w = np.arange(1, V + 1, dtype=np.float64) ** (-a)
    c = np.cumsum(w)
    return c / c[-1]


def _zipf_distinct(rng, N, K, V, a=1.1):
    cdf = zipf_cdf(V, a)

    def draw(shape):
        v = np.searchsorted(cdf, rng.random(shape), side="right")
        return np.minimum(v, V - 1).astype(np.int64)

    return _make_distinct(draw((N, K)), lambda n: draw(n))


def _student_topk_perturbed(rng, h_bits, W_bits, rows, K, V, p_replace=0.10, block=512):
    """Student's own top-K ids (descending fp64 logit) with seeded +-10 % replacement."""
    Wf = bf16_bits_to_f64(W_bits)
    out = np.empty((len(rows), K), dtype=np.int64)
    for b0 in range(0, len(rows), block):
        rb = rows[b0:b0 + block]
        z = bf16_bits_to_f64(h_bits[rb]) @ Wf.T
        out[b0:b0 + len(rb)] = np.argsort(-z, axis=1, kind="stable")[:, :K]
    replace = rng.random(out.shape) < p_replace
    rr, cc = np.nonzero(replace)
    for r, c in zip(rr.tolist(), cc.tolist()):
        row = out[r]
        while True:
            v = int(rng.integers(0, V))
            if not (row == v).any():
                row[c] = v
                break
    return out


def make_inputs(N: int, d: int, V: int, K: int, T: float = 1.0, pad_frac: float = 0.05,
                index: str = "uniform", seed: int = BASE_SEED,
                n_pad: Optional[int] = None) -> dict:
    """Draw one workload. Returns numpy arrays:
    h [N,d] uint16 (bf16 bits), W [V,d] uint16, idx [N,K] int32, t [N,K] float32,
    mask [N] uint8 (1 = valid, 0 = padding) and the scalar T."""
    rng = np.random.Generator(np.random.PCG64(seed))
    h = _normals_bf16(rng, N, d, 1.0)
    W = _normals_bf16(rng, V, d, 1.0 / np.sqrt(d))
    t = 3.0 * rng.standard_normal((N, K), dtype=np.float32)
    t = -np.sort(-t, axis=1)
    if index == "uniform":
        idx = _uniform_distinct(rng, N, K, V)
    elif index == "zipf1.1":
        idx = _zipf_distinct(rng, N, K, V, 1.1)
    elif index == "half-student":
        idx = _uniform_distinct(rng, N, K, V)
        rows = np.sort(rng.permutation(N)[: N // 2])
        idx[rows] = _student_topk_perturbed(rng, h, W, rows, K, V)
    else:
        raise ValueError(f"unknown index distribution {index!r}")
    if n_pad is None:
        n_pad = int(round(pad_frac * N))
    mask = np.ones(N, dtype=np.uint8)
    mask[rng.permutation(N)[:n_pad]] = 0
    return dict(h=h, W=W, idx=idx.astype(np.int32), t=t.astype(np.float32), mask=mask,
                T=float(T), N=N, d=d, V=V, K=K, seed=seed)


def config_inputs(i: int) -> dict:
    c = CONFIGS[i]
    x = make_inputs(c.N, c.d, c.V, c.K, c.T, c.pad_frac, c.index, config_seed(i))
    x["name"] = c.name
    return x


def fingerprint(x: dict) -> str:
    """Short digest of a workload's arrays (detects generator drift between machines)."""
    m = hashlib.sha256()
    for k in ("h", "W", "idx", "t", "mask"):
        a = np.ascontiguousarray(x[k])
        m.update(k.encode())
        m.update(a[:64].tobytes())
        m.update(a[-64:].tobytes())
        m.update(str(a.shape).encode())
    return m.hexdigest()[:16]
