"""Pins for the fp64 oracle: checks against facts fixed by the mathematics, library
routines and the pages, not against the oracle itself.

Every pin takes the oracle module as an argument so that the mutation tests can
run the same pins against deliberately broken copies of the oracle.
"""
from __future__ import annotations

import json
import os

import numpy as np
import scipy.special
import scipy.stats
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rand_problem(seed, N, d, V, K, T=1.0, pad=1, scale_w=None, overlap=False):
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((N, d))
    W = rng.standard_normal((V, d)) * (scale_w if scale_w is not None else 1.0 / np.sqrt(d))
    idx = np.stack([rng.choice(V, K, replace=False) for _ in range(N)]).astype(np.int32)
    if overlap:  # teacher ids = the student's own top-K for half the rows
        z = h @ W.T
        top = np.argsort(-z, axis=1)[:, :K]
        idx[: N // 2] = top[: N // 2]
    t = -np.sort(-3.0 * rng.standard_normal((N, K)), axis=1)
    mask = np.ones(N, dtype=np.uint8)
    mask[rng.permutation(N)[:pad]] = 0
    return h, W, idx, t, mask, T


# (P1) KL_i >= 0 for every row (Gibbs' inequality: with distinct indices the
# student's mass on the K cached ids is at most 1).
def pin_kl_nonnegative(orc):
    for seed, T in ((1, 1.0), (2, 2.0), (3, 0.5)):
        h, W, idx, t, mask, _ = _rand_problem(seed, 48, 16, 97, 9, overlap=True)
        out = orc.forward(h, W, idx, t, mask, T)
        assert np.all(out["kl"] >= -1e-12), out["kl"].min()
        assert out["loss"] >= 0.0


# (P2) KL = 0 when the student puts exactly p on the K ids and vanishing mass
# elsewhere.  W = identity (d = V) makes z = h, so the logits can be set directly.
def pin_zero_case(orc):
    rng = np.random.default_rng(7)
    for T in (1.0, 2.0, 0.7):
        N, V, K = 6, 40, 5
        t = -np.sort(-3.0 * rng.standard_normal((N, K)), axis=1)
        idx = np.stack([rng.choice(V, K, replace=False) for _ in range(N)])
        p = scipy.special.softmax(t / T, axis=1)  # library softmax
        C = 3.25
        h = np.full((N, V), -1e4 * T)
        for i in range(N):
            h[i, idx[i]] = T * np.log(p[i]) + C
        out = orc.forward(h, np.eye(V), idx, t, None, T)
        assert np.all(np.abs(out["kl"]) < 1e-12), out["kl"]
        assert abs(out["loss"]) < 1e-12


# (P3) The loss does not depend on how rows are chunked.
def pin_chunk_invariance(orc):
    h, W, idx, t, mask, T = _rand_problem(11, 70, 24, 131, 7, pad=5)
    ref = orc.forward(h, W, idx, t, mask, 1.5, row_block=70)
    g_ref = orc.backward(h, W, idx, t, mask, 1.5, row_block=70)
    for rb in (1, 7, 64):
        out = orc.forward(h, W, idx, t, mask, 1.5, row_block=rb)
        assert abs(out["loss"] - ref["loss"]) <= 1e-13 * abs(ref["loss"])
        np.testing.assert_allclose(out["lse"], ref["lse"], rtol=1e-14, atol=0)
        g = orc.backward(h, W, idx, t, mask, 1.5, row_block=rb)
        np.testing.assert_allclose(g["dh"], g_ref["dh"], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(g["dW"], g_ref["dW"], rtol=1e-12, atol=1e-15)


# (P4) A constant output bias (a ones column in h and a constant column in W)
# shifts every logit of a row equally and leaves the loss and the gradients of
# the original coordinates unchanged.
def pin_bias_shift(orc):
    h, W, idx, t, mask, T = _rand_problem(13, 33, 12, 77, 6, pad=3)
    base = orc.forward(h, W, idx, t, mask, 2.0)
    gb = orc.backward(h, W, idx, t, mask, 2.0)
    for c in (-4.0, 0.37, 9.0):
        h1 = np.concatenate([h, np.ones((h.shape[0], 1))], axis=1)
        W1 = np.concatenate([W, np.full((W.shape[0], 1), c)], axis=1)
        out = orc.forward(h1, W1, idx, t, mask, 2.0)
        assert abs(out["loss"] - base["loss"]) <= 1e-12 * abs(base["loss"])
        np.testing.assert_allclose(out["lse"] - c / 2.0, base["lse"], rtol=0, atol=1e-12)
        g = orc.backward(h1, W1, idx, t, mask, 2.0)
        np.testing.assert_allclose(g["dh"][:, :-1], gb["dh"], rtol=1e-9, atol=1e-13)
        np.testing.assert_allclose(g["dW"][:, :-1], gb["dW"], rtol=1e-9, atol=1e-13)


# (P5) Gradients agree with central finite differences of the loss.
def pin_finite_differences(orc):
    for T in (1.0, 2.0):
        h, W, idx, t, mask, _ = _rand_problem(17, 5, 4, 9, 3, pad=1, scale_w=0.8)
        g = orc.backward(h, W, idx, t, mask, T)
        eps = 1e-6

        def L(hh, WW):
            return orc.forward(hh, WW, idx, t, mask, T)["loss"]

        fd_h = np.zeros_like(h)
        for i in range(h.shape[0]):
            for j in range(h.shape[1]):
                hp, hm = h.copy(), h.copy()
                hp[i, j] += eps
                hm[i, j] -= eps
                fd_h[i, j] = (L(hp, W) - L(hm, W)) / (2 * eps)
        fd_W = np.zeros_like(W)
        for v in range(W.shape[0]):
            for j in range(W.shape[1]):
                Wp, Wm = W.copy(), W.copy()
                Wp[v, j] += eps
                Wm[v, j] -= eps
                fd_W[v, j] = (L(h, Wp) - L(h, Wm)) / (2 * eps)
        scale = max(np.abs(fd_h).max(), np.abs(fd_W).max())
        assert np.abs(g["dh"] - fd_h).max() <= 1e-7 * scale, np.abs(g["dh"] - fd_h).max()
        assert np.abs(g["dW"] - fd_W).max() <= 1e-7 * scale, np.abs(g["dW"] - fd_W).max()


# (P6a) K = 1: p = 1, so the loss is T^2 times the mean cross-entropy of z/T at
# the cached id -- torch's cross_entropy, with autograd for the gradients.
def pin_k1_cross_entropy(orc):
    for T in (1.0, 2.0):
        h, W, idx, t, mask, _ = _rand_problem(19, 64, 32, 257, 1, pad=4)
        out = orc.forward(h, W, idx, t, mask, T)
        g = orc.backward(h, W, idx, t, mask, T)
        ht = torch.tensor(h, dtype=torch.float64, requires_grad=True)
        Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
        keep = torch.tensor(mask != 0)
        ce = F.cross_entropy((ht @ Wt.T)[keep] / T, torch.tensor(idx[:, 0], dtype=torch.long)[keep])
        loss = T * T * ce
        loss.backward()
        assert abs(out["loss"] - loss.item()) <= 1e-12 * abs(loss.item())
        np.testing.assert_allclose(g["dh"], ht.grad.numpy(), rtol=1e-10, atol=1e-14)
        np.testing.assert_allclose(g["dW"], Wt.grad.numpy(), rtol=1e-10, atol=1e-14)


# (P6b) The hand-derived dz = T (q - s)/N_valid against torch autograd through
# log_softmax and kl_div (library routines), at the tiny workload's shape class.
def pin_autograd_general_k(orc):
    h, W, idx, t, mask, _ = _rand_problem(23, 96, 48, 515, 16, pad=5, overlap=True)
    T = 2.0
    g = orc.backward(h, W, idx, t, mask, T)
    out = orc.forward(h, W, idx, t, mask, T)
    ht = torch.tensor(h, dtype=torch.float64, requires_grad=True)
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    logq = torch.log_softmax((ht @ Wt.T) / T, dim=1)
    logq_k = logq.gather(1, torch.tensor(idx, dtype=torch.long))
    p = torch.softmax(torch.tensor(t, dtype=torch.float64) / T, dim=1)
    kl_rows = F.kl_div(logq_k, p, reduction="none").sum(dim=1)
    keep = torch.tensor(mask != 0, dtype=torch.float64)
    loss = T * T * (kl_rows * keep).sum() / keep.sum()
    loss.backward()
    assert abs(out["loss"] - loss.item()) <= 1e-12 * abs(loss.item())
    np.testing.assert_allclose(g["dh"], ht.grad.numpy(), rtol=1e-9, atol=1e-14)
    np.testing.assert_allclose(g["dW"], Wt.grad.numpy(), rtol=1e-9, atol=1e-14)


# (P7) sum_v dz_iv = T (sum_v q - sum_k p)/N_valid = 0 for each row, hence the
# rows of dW sum to the zero vector.
def pin_zero_sum(orc):
    h, W, idx, t, mask, T = _rand_problem(29, 40, 20, 300, 12, pad=2)
    g = orc.backward(h, W, idx, t, mask, 1.0)
    col = g["dW"].sum(axis=0)
    assert np.abs(col).max() <= 1e-13 * max(1.0, np.abs(g["dW"]).max() * W.shape[0])


# (P8) Closed form: W = 0 makes q uniform, lse = log V and
# KL_i = log V - entropy(p_i) (scipy's entropy).
def pin_uniform_student(orc):
    for T in (1.0, 3.0):
        h, W, idx, t, mask, _ = _rand_problem(31, 25, 8, 1000, 10, pad=2)
        W = np.zeros_like(W)
        out = orc.forward(h, W, idx, t, mask, T)
        np.testing.assert_allclose(out["lse"], np.log(1000.0), rtol=0, atol=1e-12)
        p = scipy.special.softmax(t / T, axis=1)
        kl = np.log(1000.0) - scipy.stats.entropy(p, axis=1)
        keep = mask != 0
        np.testing.assert_allclose(out["kl"], kl, rtol=1e-12, atol=1e-12)
        assert abs(out["loss"] - T * T * kl[keep].mean()) <= 1e-12 * abs(out["loss"])


# (P9) lse is scipy's logsumexp of z/T.
def pin_lse_library(orc):
    h, W, idx, t, mask, T = _rand_problem(37, 20, 10, 333, 4)
    for T in (1.0, 0.25, 4.0):
        out = orc.forward(h, W, idx, t, mask, T)
        np.testing.assert_allclose(out["lse"], scipy.special.logsumexp((h @ W.T) / T, axis=1),
                                   rtol=1e-14, atol=1e-13)


# (P10) The page's soft-label example: logs of the printed probabilities as the
# cached logits give back the renormalised probabilities, softened by T.
def pin_page_soft_labels(orc):
    with open(os.path.join(GOLDEN, "soft_labels_ml_book.json")) as f:
        g = json.load(f)
    pp = np.array(g["p_printed"])
    t = np.log(pp)[None, :]
    p1, ok = orc.teacher_distribution(t, 1.0)
    assert ok.all()
    np.testing.assert_allclose(p1[0], pp / 0.99, rtol=1e-14)
    for T in (3.0, 5.0):
        pT, _ = orc.teacher_distribution(t, T)
        ref = pp ** (1.0 / T)
        np.testing.assert_allclose(pT[0], ref / ref.sum(), rtol=1e-13)
        assert pT[0, 0] < p1[0, 0] and pT[0, -1] > p1[0, -1]  # softened


# (P11) Degenerate rows: -inf teacher logits carry p = 0; a row with all -inf
# or mask 0 does not count; N_valid = 0 gives a zero loss and zero gradients.
def pin_degenerate_rows(orc):
    h, W, idx, t, mask, T = _rand_problem(41, 12, 6, 50, 5, pad=0)
    t = t.copy()
    t[0, 3:] = -np.inf
    t[1, :] = -np.inf
    p, has = orc.teacher_distribution(t, 1.0)
    assert not has[1] and has[0] and np.all(p[1] == 0) and np.all(p[0, 3:] == 0)
    np.testing.assert_allclose(p[0, :3], scipy.special.softmax(t[0, :3]), rtol=1e-14)
    out = orc.forward(h, W, idx, t, mask, 1.0)
    assert out["n_valid"] == 11 and np.isfinite(out["loss"])
    keep = np.ones(12, bool)
    keep[1] = False
    ref = orc.forward(h[keep], W, idx[keep], t[keep], mask[keep], 1.0)
    assert abs(out["loss"] - ref["loss"]) <= 1e-13 * abs(ref["loss"])
    zero = orc.forward(h, W, idx, t, np.zeros(12, np.uint8), 1.0)
    gz = orc.backward(h, W, idx, t, np.zeros(12, np.uint8), 1.0)
    assert zero["loss"] == 0.0 and zero["n_valid"] == 0
    assert not gz["dh"].any() and not gz["dW"].any()


# (P12) Sampled-row and sampled-column helpers agree with the full pass.
def pin_sampled_helpers(orc):
    h, W, idx, t, mask, T = _rand_problem(43, 50, 16, 211, 8, pad=4)
    full = orc.forward(h, W, idx, t, mask, 1.5)
    g = orc.backward(h, W, idx, t, mask, 1.5, grad_loss=0.75)
    rows = np.array([0, 3, 17, 49])
    s = orc.rows_forward_backward(h, W, idx, t, mask, 1.5, rows, grad_loss=0.75)
    np.testing.assert_allclose(s["lse"], full["lse"][rows], rtol=1e-14)
    np.testing.assert_allclose(s["kl"], full["kl"][rows], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(s["dh"], g["dh"][rows], rtol=1e-12, atol=1e-16)
    vr = np.array([0, 5, int(idx[3, 2]), 210])
    dw = orc.dW_rows(h, W, idx, t, mask, 1.5, full["lse"], vr, grad_loss=0.75, row_block=13)
    np.testing.assert_allclose(dw, g["dW"][vr], rtol=1e-11, atol=1e-16)
    np.testing.assert_allclose(orc.student_lse(h, W, 1.5, row_block=9), full["lse"], rtol=1e-14)


# (T1) Teacher cache, closed form: with W = I (d = V) the logits are h itself, so
# the cache is the K largest entries of each h row -- numpy's stable argsort of -h.
def pin_topk_identity_head(orc):
    rng = np.random.default_rng(53)
    V = 300
    h = rng.standard_normal((9, V))
    for K in (1, 7, 100, V):
        idx, val, _ = orc.teacher_topk(h, np.eye(V), K)
        ref = np.argsort(-h, axis=1, kind="stable")[:, :K]
        assert np.array_equal(idx, ref)
        np.testing.assert_array_equal(val, np.take_along_axis(h, ref, axis=1))


# (T2) Ties go to the smaller id, and the order is by logit first: duplicated
# vocabulary rows give equal logits; a permutation of W's rows permutes the ids.
def pin_topk_ties_and_permutation(orc):
    rng = np.random.default_rng(59)
    d, V, K = 6, 50, 12
    h = rng.standard_normal((5, d))
    W = rng.standard_normal((V, d))
    W[30] = W[4]
    W[41] = W[4]
    W[17] = W[2]
    idx, val, _ = orc.teacher_topk(h, W, V)
    assert np.all(np.diff(val, axis=1) <= 0)
    for i in range(5):
        pos = {int(v): k for k, v in enumerate(idx[i])}
        assert pos[4] < pos[30] < pos[41] and pos[2] < pos[17]
        assert val[i, pos[4]] == val[i, pos[41]]
    perm = rng.permutation(V)
    idx_p, val_p, _ = orc.teacher_topk(h, W[perm], K)
    z = h @ W.T
    for i in range(5):  # the same K logits; each id names the permuted row it came from
        np.testing.assert_allclose(val_p[i], val[i, :K], rtol=1e-14)
        np.testing.assert_allclose(val_p[i], z[i, perm[idx_p[i]]], rtol=1e-14)


# (M1) The KL + cross-entropy mixture against torch autograd through log_softmax,
# kl_div and cross_entropy (library routines), for several alpha and T; alpha = 1
# is the plain loss and alpha = 0 plain cross-entropy.
def pin_mixture_autograd(orc):
    if not hasattr(orc, "forward_mix"):
        return  # only the numpy oracle carries the mixture
    h, W, idx, t, mask, _ = _rand_problem(61, 48, 24, 211, 8, pad=3, overlap=True)
    label = np.random.default_rng(62).integers(0, 211, 48)
    for T, alpha in ((1.0, 0.5), (2.0, 0.3), (3.0, 1.0), (1.5, 0.0)):
        out = orc.forward_mix(h, W, idx, t, mask, label, T, alpha)
        g = orc.backward_mix(h, W, idx, t, mask, label, T, alpha, grad_loss=0.7)
        ht = torch.tensor(h, dtype=torch.float64, requires_grad=True)
        Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
        z = ht @ Wt.T
        logq = torch.log_softmax(z / T, dim=1).gather(1, torch.tensor(idx, dtype=torch.long))
        p = torch.softmax(torch.tensor(t, dtype=torch.float64) / T, dim=1)
        keep = torch.tensor(mask != 0)
        kl = F.kl_div(logq, p, reduction="none").sum(dim=1)[keep].mean()
        ce = F.cross_entropy(z[keep], torch.tensor(label, dtype=torch.long)[keep])
        loss = alpha * T * T * kl + (1 - alpha) * ce
        (0.7 * loss).backward()
        assert abs(out["loss"] - loss.item()) <= 1e-12 * abs(loss.item())
        np.testing.assert_allclose(g["dh"], ht.grad.numpy(), rtol=1e-9, atol=1e-14)
        np.testing.assert_allclose(g["dW"], Wt.grad.numpy(), rtol=1e-9, atol=1e-14)
        if alpha == 1.0:
            plain = orc.forward(h, W, idx, t, mask, T)
            assert abs(plain["loss"] - out["loss"]) <= 1e-13 * abs(plain["loss"])


# (M2) Mixture gradients against central finite differences of its loss.
def pin_mixture_finite_differences(orc):
    if not hasattr(orc, "forward_mix"):
        return
    h, W, idx, t, mask, _ = _rand_problem(67, 4, 3, 8, 3, pad=1, scale_w=0.8)
    label = np.array([5, 0, 7, 2])
    T, alpha, eps = 2.0, 0.4, 1e-6
    g = orc.backward_mix(h, W, idx, t, mask, label, T, alpha)

    def L(hh, WW):
        return orc.forward_mix(hh, WW, idx, t, mask, label, T, alpha)["loss"]

    for A, G, f in ((h, g["dh"], lambda a: L(a, W)), (W, g["dW"], lambda a: L(h, a))):
        fd = np.zeros_like(A)
        for i in range(A.shape[0]):
            for j in range(A.shape[1]):
                ap, am = A.copy(), A.copy()
                ap[i, j] += eps
                am[i, j] -= eps
                fd[i, j] = (f(ap) - f(am)) / (2 * eps)
        assert np.abs(G - fd).max() <= 1e-7 * max(1.0, np.abs(fd).max())


ALL_PINS = [
    pin_kl_nonnegative, pin_zero_case, pin_chunk_invariance, pin_bias_shift,
    pin_finite_differences, pin_k1_cross_entropy, pin_autograd_general_k, pin_zero_sum,
    pin_uniform_student, pin_lse_library, pin_page_soft_labels, pin_degenerate_rows,
    pin_sampled_helpers, pin_topk_identity_head, pin_topk_ties_and_permutation,
    pin_mixture_autograd, pin_mixture_finite_differences,
]
