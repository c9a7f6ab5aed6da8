"""Plain fp64 CPU oracle for the fused top-K forward-KL distillation loss.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only the tests, the package smoke check and the benchmark's CPU-baseline leg
may call it.  It shares no code with the CUDA library.

What it computes (the plain definition, with a library matmul as one step):

* Teacher cache.  Each token keeps K (index, logit) pairs of the teacher
  ("Effektivnaya distillyatsiya znaniy", malakhovai.ru, paragraph 2: the top-100
  per position are cached offline; "Wissensdestillation mit deutlich weniger
  GPU-Speicher", dailytechsnack.ch, section "Teacher-Ausgaben einmalig
  zwischenspeichern").  The teacher distribution is the softmax of t/T taken
  over those K entries, i.e. renormalised over the cache (temperature: "Distillyatsiya
  i szhatie modeley", ml-book.com, section "Kak eto rabotaet: myagkie metki i
  temperatura" -- logits are divided by T before the softmax).
* Student.  z = h W^T over the FULL vocabulary, a = z/T, lse_i = logsumexp_v a_iv,
  log q_iv = a_iv - lse_i.
* Loss.  Forward KL per token, KL_i = sum_k p_ik (log p_ik - log q_{i,idx_ik}),
  with 0 log 0 = 0; loss = T^2 * sum_{valid i} KL_i / N_valid (the T^2 factor
  restores the gradient scale that the temperature shrinks: same ml-book.com
  section, last paragraph).  N_valid = 0 gives loss 0.
* Gradients.  dz_iv = valid_i * g * T * (q_iv - s_iv) / N_valid with
  s_iv = sum_{k: idx_ik = v} p_ik and g the upstream gradient; dh = dz W and
  dW = dz^T h.

A token is valid when its mask byte is non-zero and at least one of its teacher
logits is finite (a row of all -inf logits carries no distribution).

The pages leave the chunking to the implementation ("Multiverse Computing
uzhala distillyatsiyu", iitak.ru, paragraph 3: chunks are added to a running
total and recomputed in the backward pass); the oracle materialises full logit
rows block by block, which is the definition itself.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "teacher_distribution", "row_valid", "student_lse", "forward", "backward",
    "rows_forward_backward", "dW_rows", "kl_rows_from_logits", "teacher_topk",
    "forward_mix", "backward_mix",
]


def teacher_distribution(tlogit: np.ndarray, T: float):
    """p = softmax_k(t/T) over the K cached logits, fp64.

    Returns (p [N,K], has_mass [N] bool).  Entries with t = -inf get p = 0; a row
    whose logits are all -inf gets p = 0 everywhere and has_mass False.
    """
    u = np.asarray(tlogit, dtype=np.float64) / float(T)
    finite = np.isfinite(u)
    has_mass = finite.any(axis=1)
    m = np.where(finite, u, -np.inf).max(axis=1)
    m = np.where(has_mass, m, 0.0)
    e = np.where(finite, np.exp(np.where(finite, u, 0.0) - m[:, None]), 0.0)
    s = e.sum(axis=1)
    p = np.where(has_mass[:, None], e / np.where(s > 0, s, 1.0)[:, None], 0.0)
    return p, has_mass


def row_valid(mask, tlogit, T):
    _, has_mass = teacher_distribution(tlogit, T)
    m = np.ones(len(has_mass), dtype=bool) if mask is None else (np.asarray(mask) != 0)
    return m & has_mass


def _logsumexp_rows(a: np.ndarray) -> np.ndarray:
    m = a.max(axis=1)
    return m + np.log(np.exp(a - m[:, None]).sum(axis=1))


def kl_rows_from_logits(z: np.ndarray, idx: np.ndarray, p: np.ndarray, T: float):
    """Per-row forward KL from a block of materialised student logits z [B,V].

    Returns (lse [B], KL [B]).  0 log 0 = 0.
    """
    a = z / float(T)
    lse = _logsumexp_rows(a)
    a_idx = np.take_along_axis(a, idx.astype(np.int64), axis=1)
    logq = a_idx - lse[:, None]
    logp = np.where(p > 0, np.log(np.where(p > 0, p, 1.0)), 0.0)
    kl = np.where(p > 0, p * (logp - logq), 0.0).sum(axis=1)
    return lse, kl


def student_lse(h, W, T, row_block=256):
    """lse_i = logsumexp_v (h_i . W_v)/T for every row, fp64."""
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    out = np.empty(h.shape[0])
    for r0 in range(0, h.shape[0], row_block):
        z = h[r0:r0 + row_block] @ W.T
        out[r0:r0 + row_block] = _logsumexp_rows(z / float(T))
    return out


def forward(h, W, idx, tlogit, mask, T, row_block=256):
    """Loss, per-row lse and per-row KL over all rows.

    h [N,d], W [V,d] (any float dtype, used in fp64), idx [N,K] ints, tlogit
    [N,K], mask [N] (non-zero = valid) or None.  Rows are processed in blocks of
    `row_block`; the per-row values do not depend on the block size.
    """
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    N = h.shape[0]
    p, _ = teacher_distribution(tlogit, T)
    valid = row_valid(mask, tlogit, T)
    lse = np.empty(N)
    kl = np.empty(N)
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        z = h[r0:r1] @ W.T
        lse[r0:r1], kl[r0:r1] = kl_rows_from_logits(z, idx[r0:r1], p[r0:r1], T)
    n_valid = int(valid.sum())
    loss = float(T) ** 2 * kl[valid].sum() / n_valid if n_valid > 0 else 0.0
    return dict(loss=loss, lse=lse, kl=kl, n_valid=n_valid, valid=valid)


def _dz_block(z, idx, p, T, coef):
    """dz for a block of rows from materialised logits; coef_i = valid_i * g * T / N_valid."""
    a = z / float(T)
    lse = _logsumexp_rows(a)
    q = np.exp(a - lse[:, None])
    s = np.zeros_like(q)
    rows = np.repeat(np.arange(z.shape[0]), idx.shape[1])
    np.add.at(s, (rows, idx.reshape(-1).astype(np.int64)), p.reshape(-1))
    return coef[:, None] * (q - s), lse


def backward(h, W, idx, tlogit, mask, T, grad_loss=1.0, row_block=256):
    """dh [N,d] and dW [V,d] (fp64) of the loss times `grad_loss`."""
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    N = h.shape[0]
    p, _ = teacher_distribution(tlogit, T)
    valid = row_valid(mask, tlogit, T)
    n_valid = int(valid.sum())
    dh = np.zeros_like(h)
    dW = np.zeros_like(W)
    if n_valid == 0:
        return dict(dh=dh, dW=dW, n_valid=0)
    coef = valid.astype(np.float64) * float(grad_loss) * float(T) / n_valid
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        z = h[r0:r1] @ W.T
        dz, _ = _dz_block(z, idx[r0:r1], p[r0:r1], T, coef[r0:r1])
        dh[r0:r1] = dz @ W
        dW += dz.T @ h[r0:r1]
    return dict(dh=dh, dW=dW, n_valid=n_valid)


def rows_forward_backward(h, W, idx, tlogit, mask, T, rows, grad_loss=1.0, row_block=128):
    """lse, KL and dh for a subset of rows (the global N_valid comes from all rows).

    Used where a full pass over every row is too slow: each sampled row needs
    one full logit row (2 d V flops) for lse/KL and one more product for dh.
    """
    rows = np.asarray(rows, dtype=np.int64)
    W = np.asarray(W, dtype=np.float64)
    p_all, _ = teacher_distribution(tlogit, T)
    valid_all = row_valid(mask, tlogit, T)
    n_valid = int(valid_all.sum())
    lse = np.empty(len(rows))
    kl = np.empty(len(rows))
    dh = np.zeros((len(rows), W.shape[1]))
    for b0 in range(0, len(rows), row_block):
        rb = rows[b0:b0 + row_block]
        z = np.asarray(h[rb], dtype=np.float64) @ W.T
        lse[b0:b0 + len(rb)], kl[b0:b0 + len(rb)] = kl_rows_from_logits(z, idx[rb], p_all[rb], T)
        if n_valid > 0:
            coef = valid_all[rb].astype(np.float64) * float(grad_loss) * float(T) / n_valid
            dz, _ = _dz_block(z, idx[rb], p_all[rb], T, coef)
            dh[b0:b0 + len(rb)] = dz @ W
    return dict(lse=lse, kl=kl, dh=dh, n_valid=n_valid)


def dW_rows(h, W, idx, tlogit, mask, T, lse, vocab_rows, grad_loss=1.0, row_block=4096):
    """dW restricted to the vocabulary rows `vocab_rows`, given lse for every token.

    dW_v = sum_i dz_iv h_i needs the logit column z_{.v} over all tokens and the
    per-token lse (from `forward` or `student_lse`).
    """
    vocab_rows = np.asarray(vocab_rows, dtype=np.int64)
    Wv = np.asarray(W[vocab_rows], dtype=np.float64)
    N = h.shape[0]
    p, _ = teacher_distribution(tlogit, T)
    valid = row_valid(mask, tlogit, T)
    n_valid = int(valid.sum())
    out = np.zeros((len(vocab_rows), Wv.shape[1]))
    if n_valid == 0:
        return out
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        hb = np.asarray(h[r0:r1], dtype=np.float64)
        a = (hb @ Wv.T) / float(T)
        q = np.exp(a - np.asarray(lse[r0:r1], dtype=np.float64)[:, None])
        # s_iv: teacher mass that row i puts on vocabulary id vocab_rows[j]
        hit = idx[r0:r1, :, None] == vocab_rows[None, None, :]
        s = (p[r0:r1, :, None] * hit).sum(axis=1)
        coef = valid[r0:r1].astype(np.float64) * float(grad_loss) * float(T) / n_valid
        out += (coef[:, None] * (q - s)).T @ hb
    return out


def teacher_topk(h, W, K, rows=None, row_block=256):
    """The teacher cache: per row the K largest logits z = h W^T (fp64) and their ids.

    Ordered by logit descending, equal logits by id ascending -- the top-100 per
    position that "Effektivnaya distillyatsiya znaniy" (malakhovai.ru, paragraph 2)
    and "Wissensdestillation mit deutlich weniger GPU-Speicher" (dailytechsnack.ch,
    section "Teacher-Ausgaben einmalig zwischenspeichern") cache once, offline.
    `rows` restricts the computation to those rows.  Returns (idx [n,K] int64,
    logit [n,K] fp64, z_full [n,V] fp64 of the same rows).
    """
    W = np.asarray(W, dtype=np.float64)
    rows = np.arange(h.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    idx = np.empty((len(rows), K), dtype=np.int64)
    val = np.empty((len(rows), K))
    zs = np.empty((len(rows), W.shape[0]))
    for b0 in range(0, len(rows), row_block):
        rb = rows[b0:b0 + row_block]
        z = np.asarray(h[rb], dtype=np.float64) @ W.T
        # sort key: logit descending, then id ascending (a stable sort of -z keeps ids ascending)
        order = np.argsort(-z, axis=1, kind="stable")[:, :K]
        idx[b0:b0 + len(rb)] = order
        val[b0:b0 + len(rb)] = np.take_along_axis(z, order, axis=1)
        zs[b0:b0 + len(rb)] = z
    return idx, val, zs


def forward_mix(h, W, idx, tlogit, mask, label, T, alpha, row_block=256):
    """KL + hard-label cross-entropy: loss = alpha T^2 mean KL_i + (1 - alpha) mean CE_i.

    "Distillyatsiya i szhatie modeley" (ml-book.com, section "Kak eto rabotaet:
    myagkie metki i temperatura"): the student's loss mixes the KL between the
    softened distributions with the ordinary cross-entropy on the true labels;
    the weights (alpha, 1 - alpha) are the usual convex mix, the page's formula
    being lost.  CE_i = lse1_i - z_{i,label_i} with lse1 the logsumexp of z at
    temperature 1; both means run over the valid rows.  Returns the forward's
    dict plus lse1 [N] and ce [N].
    """
    out = forward(h, W, idx, tlogit, mask, T, row_block)
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    label = np.asarray(label, dtype=np.int64)
    N = h.shape[0]
    lse1 = np.empty(N)
    ce = np.empty(N)
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        z = h[r0:r1] @ W.T
        lse1[r0:r1] = _logsumexp_rows(z)
        ce[r0:r1] = lse1[r0:r1] - z[np.arange(r1 - r0), label[r0:r1]]
    valid, n_valid = out["valid"], out["n_valid"]
    if n_valid > 0:
        kl_mean = out["kl"][valid].sum() / n_valid
        ce_mean = ce[valid].sum() / n_valid
        out["loss"] = float(alpha) * float(T) ** 2 * kl_mean + (1.0 - float(alpha)) * ce_mean
    out["lse1"] = lse1
    out["ce"] = ce
    return out


def backward_mix(h, W, idx, tlogit, mask, label, T, alpha, grad_loss=1.0, row_block=256):
    """dh, dW of forward_mix's loss times grad_loss:
    dz_iv = g valid_i [alpha T (q_iv - s_iv) + (1 - alpha)(q1_iv - [v = label_i])] / N_valid."""
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    label = np.asarray(label, dtype=np.int64)
    N = h.shape[0]
    p, _ = teacher_distribution(tlogit, T)
    valid = row_valid(mask, tlogit, T)
    n_valid = int(valid.sum())
    dh = np.zeros_like(h)
    dW = np.zeros_like(W)
    if n_valid == 0:
        return dict(dh=dh, dW=dW, n_valid=0)
    coef = valid.astype(np.float64) * float(grad_loss) / n_valid
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        z = h[r0:r1] @ W.T
        kl_part, _ = _dz_block(z, idx[r0:r1], p[r0:r1], T, coef[r0:r1] * float(T) * float(alpha))
        q1 = np.exp(z - _logsumexp_rows(z)[:, None])
        q1[np.arange(r1 - r0), label[r0:r1]] -= 1.0
        dz = kl_part + (coef[r0:r1] * (1.0 - float(alpha)))[:, None] * q1
        dh[r0:r1] = dz @ W
        dW += dz.T @ h[r0:r1]
    return dict(dh=dh, dW=dW, n_valid=n_valid)
