"""Plain float64 CPU oracle for the fused-linear Jensen-Shannon distillation loss.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it. It shares no code with the CUDA library.

What it computes, and the passages it follows (Liger-Kernel pull requests):

* "[Perf] Fuse log-softmax into fused_linear_jsd kernel" (PR 1352), "Details":
  the student and teacher logits are the two GEMMs X_s W_s^T and X_t W_t^T; both
  log-softmaxes are taken on the temperature-scaled logits; the per-row loss
  is a sum over V (loss_1d has shape (BT,)); the gradient with respect to the
  log-probabilities X (dX) is pushed through the log-softmax Jacobian with the
  cross-column term dX_sum, and the result is the gradient of the student
  logits.
* Same page, "Testing Done": the beta branches -- 0.0 is forward KL, 0.1 and
  0.5 are the generalized JSD, 1.0 is reverse KL.
* Same page, "Open questions" 2: the temperature divides the logits once; no
  T^2 factor anywhere.
* "Fix TVD gradient at p == q" (PR 1374), "Summary": a distance whose
  per-element derivative is zero at p == q must give an exactly zero
  gradient there; transferred to the JSD as an exactly zero per-element
  contribution where the student and teacher log-probabilities tie.
* "perf(flce): write the weight-gradient product directly into grad_weight"
  (PR 1429), "Summary": grad_weight is the sum over row chunks of
  dlogits^T . X_s.

Readings where the pages are silent (each is listed with its reason in the
design notes of the repository):

* P is the teacher distribution, Q the student one. X = log Q, Y = log P.
  beta = 0 gives KL(P||Q), beta = 1 gives KL(Q||P), and 0 < beta < 1 gives
  beta*KL(P||M) + (1-beta)*KL(Q||M) with M = beta*P + (1-beta)*Q.
* The endpoints are exact compares (beta == 0.0, beta == 1.0).
* Reductions: sum (w = 1), batchmean (w = 1/n, n = rows whose label is not
  ignore_index), mean (w = 1/(n*V)), none (per-row vector, the gradient is
  that of sum_r row_grad[r]*L_r). With n == 0 the loss and every gradient are 0.
* Rows whose label equals ignore_index contribute 0 to the loss and have a
  zero gradient.
* The tie rule sets the per-element loss to 0 in every branch where X_j == Y_j
  exactly, and also the per-element log-probability gradient of the
  generalized branch (whose exact value is 0 there). The endpoint branches
  use closed-form logit gradients (Q - P at beta = 0, Q*(X - Y - L) at
  beta = 1), which are exactly what the calculus gives at a tie.

Every array is float64. Inputs are the exact values of the bf16/fp32 tensors,
widened to float64.
"""
from __future__ import annotations

import numpy as np

REDUCTIONS = ("none", "sum", "mean", "batchmean")


# ---------------------------------------------------------------------------
# bf16 rounding (diagnostic only)
# ---------------------------------------------------------------------------
def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 value, ties to even, and widen to float64.

    Used only by the ``emulate_rounding`` diagnostic: the fused kernel stores the
    GEMM output in the input dtype ("Open questions" 1 of PR 1352) and writes
    dlogits over the student logits buffer ("Details" of PR 1352), so with
    bf16 inputs both round to bf16. The value is first rounded to float32
    (nearest), then to bfloat16 (nearest, ties to even) by integer arithmetic
    on the float32 bit pattern. NaN and infinity are not expected here.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lower = u & np.uint64(0xFFFF)
    upper = u >> np.uint64(16)
    half = np.uint64(0x8000)
    round_up = (lower > half) | ((lower == half) & ((upper & np.uint64(1)) == np.uint64(1)))
    upper = upper + round_up.astype(np.uint64)
    out = (upper << np.uint64(16)).astype(np.uint32).view(np.float32)
    return out.astype(np.float64)


def _store_round(x: np.ndarray, mode) -> np.ndarray:
    """Round to the storage dtype named by ``mode`` (True/"bf16" or "fp32")."""
    if mode == "fp32":
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
    return bf16_round(x)


# ---------------------------------------------------------------------------
# the two logits GEMMs
# ---------------------------------------------------------------------------
def logits(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """z = x . w^T for x [rows x H] and the lm_head weight w [V x H] (PR 1352,
    "Summary": the logits are the product of hidden states and lm_head weight)."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T


def log_softmax_rows(a: np.ndarray) -> np.ndarray:
    """Row-wise log-softmax a - logsumexp(a), with the max subtracted first."""
    m = np.max(a, axis=1, keepdims=True)
    lse = m + np.log(np.sum(np.exp(a - m), axis=1, keepdims=True))
    return a - lse


# ---------------------------------------------------------------------------
# per-row JSD and its gradient with respect to the scaled student logits
# ---------------------------------------------------------------------------
def tie_mask(z_s: np.ndarray, z_t: np.ndarray, temperature: float) -> np.ndarray:
    """Elements where the student and teacher log-probabilities are exactly
    equal, X_j == Y_j (the tie rule of PR 1374 "Summary": such an element
    contributes exactly zero). Shape [rows x V], boolean."""
    a = np.asarray(z_s, dtype=np.float64) / temperature
    b = np.asarray(z_t, dtype=np.float64) / temperature
    return log_softmax_rows(a) == log_softmax_rows(b)


def zero_masks(z_s, z_t, labels, beta: float, temperature: float, ignore_index: int = -100):
    """Where the method itself gives exact zeros (not where a float result
    happens to cancel), for rows whose logits are z_s, z_t.

    Returns (loss_zero [rows], dz_zero [rows x V]):
    * ignored rows: loss 0 and dlogits 0 (reading of ignore_index);
    * rows tied at every element: every per-element loss is 0, so L = 0, and
      the logit gradient is 0 in every branch (beta = 0: Q - P = 0; beta = 1:
      Q (X - Y - L) = 0; generalized: dX = 0 at every element, so dX_sum = 0);
    * beta = 0: dlogits (Q - P) / T is exactly 0 at every tied element of any
      row, since Q == P there (PR 1374 "Summary" carried to the logit gradient
      by PR 1352 "Details"). In the other branches a tied element of an
      untied row has the nonzero gradient -Q_j L (beta = 1) or -Q_j dX_sum.
    """
    tie = tie_mask(z_s, z_t, temperature)
    rows = tie.shape[0]
    valid = np.ones(rows, dtype=bool) if labels is None else \
        np.asarray(labels).reshape(-1) != ignore_index
    full = np.all(tie, axis=1)
    loss_zero = ~valid | full
    dz_zero = np.zeros_like(tie)
    if beta == 0.0:
        dz_zero |= tie
    dz_zero[loss_zero] = True
    return loss_zero, dz_zero


def jsd_rows(z_s: np.ndarray, z_t: np.ndarray, beta: float, temperature: float):
    """Per-row loss L_r (shape [rows]) and dA = dL_r/da (shape [rows x V]).

    a = z_s / T and b = z_t / T are the scaled logits (PR 1352, "Open
    questions" 2: divide once). X = log_softmax(a) is the student log-prob
    (log Q), Y = log_softmax(b) the teacher log-prob (log P). The branches
    follow PR 1352 "Testing Done" (0.0 forward KL, 1.0 reverse KL, otherwise
    generalized). For the generalized branch, dX_j = (1-beta) Q_j (X_j - log M_j)
    is the gradient with respect to the log-prob and the logit gradient is
    dX_j - Q_j * dX_sum (PR 1352, "Details": dX_sum is a cross-column term).
    The tie rule of PR 1374 "Summary" zeroes the per-element contribution
    where X_j == Y_j.
    """
    if temperature <= 0:
        raise ValueError("temperature must be > 0")
    if not (0.0 <= beta <= 1.0):
        raise ValueError("beta must be in [0, 1]")
    a = np.asarray(z_s, dtype=np.float64) / temperature
    b = np.asarray(z_t, dtype=np.float64) / temperature
    X = log_softmax_rows(a)
    Y = log_softmax_rows(b)
    Q = np.exp(X)
    P = np.exp(Y)
    tie = X == Y  # the same test as tie_mask
    if beta == 0.0:
        # forward KL(P || Q)
        ell = np.where(tie, 0.0, P * (Y - X))
        L = ell.sum(axis=1)
        dA = Q - P
    elif beta == 1.0:
        # reverse KL(Q || P)
        ell = np.where(tie, 0.0, Q * (X - Y))
        L = ell.sum(axis=1)
        dA = Q * (X - Y - L[:, None])
    else:
        M = beta * P + (1.0 - beta) * Q
        # where P and Q both underflow to 0 the terms are 0 * log 0 = 0
        zero = tie | (M == 0.0)
        logM = np.log(np.where(M == 0.0, 1.0, M))
        ell = beta * P * (Y - logM) + (1.0 - beta) * Q * (X - logM)
        ell = np.where(zero, 0.0, ell)
        dX = np.where(zero, 0.0, (1.0 - beta) * Q * (X - logM))
        L = ell.sum(axis=1)
        dX_sum = dX.sum(axis=1)
        dA = dX - Q * dX_sum[:, None]
    return L, dA


# ---------------------------------------------------------------------------
# the whole fused-linear JSD forward + backward
# ---------------------------------------------------------------------------
def row_weights(labels, bt: int, v: int, reduction: str, ignore_index: int = -100,
                row_grad=None):
    """Per-row loss weights w_r and the valid-row count n.

    Reading of the reductions (the pages name four reductions in PR 1374
    "Details" and pin "batchmean" as division by the row count in the tie
    table of PR 1374): sum -> 1, batchmean -> 1/n, mean -> 1/(n*V),
    none -> row_grad[r] (1 when absent). Ignored rows get weight 0.
    """
    if reduction not in REDUCTIONS:
        raise ValueError(f"unknown reduction {reduction!r}")
    if labels is None:
        valid = np.ones(bt, dtype=bool)
    else:
        valid = np.asarray(labels).reshape(-1) != ignore_index
    n = int(valid.sum())
    if reduction == "none":
        rg = np.ones(bt) if row_grad is None else np.asarray(row_grad, dtype=np.float64)
        w = np.where(valid, rg, 0.0)
    elif n == 0:
        w = np.zeros(bt)
    elif reduction == "sum":
        w = valid.astype(np.float64)
    elif reduction == "batchmean":
        w = valid / float(n)
    else:  # mean
        w = valid / (float(n) * float(v))
    return w, valid, n


def fljsd_ref(x_s, w_s, x_t, w_t, labels=None, *, beta: float = 0.5,
              temperature: float = 1.0, reduction: str = "batchmean",
              ignore_index: int = -100, row_grad=None, emulate_rounding: bool = False,
              block_rows: int = 256, t2_scale: bool = False):
    """Loss, grad_input (d/dX_s) and grad_weight (d/dW_s) of the fused-linear JSD.

    Rows are processed in blocks of ``block_rows`` only to bound memory; each row
    is independent of the others except through the valid-row count n.
    grad_weight is the sum over blocks of dz^T . X_s (PR 1429, "Summary").

    With ``emulate_rounding`` the logits and dlogits are rounded to the input
    dtype as the kernels store them (PR 1352, "Open questions" 1: the GEMM
    output keeps the input dtype; "Details": dlogits overwrite the logits
    buffer): True or "bf16" rounds to bfloat16, "fp32" to float32. It is a
    diagnostic for cases where 1/T magnifies the storage rounding, not the
    definition.

    ``t2_scale`` multiplies the loss and both gradients by T^2 (the opt-in
    Hinton et al. 2015 scaling that PR 1352, "Open questions" 2, discusses; off
    by default, as on the pages).

    Returns (loss, grad_input, grad_weight): loss is a float for sum, mean and
    batchmean, and a [BT] array for none.
    """
    x_s = np.asarray(x_s, dtype=np.float64)
    w_s = np.asarray(w_s, dtype=np.float64)
    x_t = np.asarray(x_t, dtype=np.float64)
    w_t = np.asarray(w_t, dtype=np.float64)
    bt = x_s.shape[0]
    v = w_s.shape[0]
    assert w_s.shape[1] == x_s.shape[1] and x_t.shape[0] == bt and w_t.shape == (v, x_t.shape[1])

    def blocks():
        for r0 in range(0, bt, block_rows):
            r1 = min(bt, r0 + block_rows)
            zs = logits(x_s[r0:r1], w_s)
            zt = logits(x_t[r0:r1], w_t)
            if emulate_rounding:
                zs, zt = _store_round(zs, emulate_rounding), _store_round(zt, emulate_rounding)
            yield r0, r1, zs, zt

    out = _from_logit_blocks(blocks(), x_s, w_s, labels, beta, temperature, reduction,
                             ignore_index, row_grad, emulate_rounding)
    if t2_scale:
        t2 = temperature * temperature
        out = (out[0] * t2, out[1] * t2, out[2] * t2)
    return out


def fljsd_from_logits(z_s, z_t, x_s, w_s, labels=None, *, beta: float = 0.5,
                      temperature: float = 1.0, reduction: str = "batchmean",
                      ignore_index: int = -100, row_grad=None, block_rows: int = 256):
    """The same as ``fljsd_ref`` for logits computed beforehand with ``logits``
    (so that one pair of logits GEMMs serves a sweep of beta, T and reduction)."""
    x_s = np.asarray(x_s, dtype=np.float64)
    w_s = np.asarray(w_s, dtype=np.float64)
    bt = x_s.shape[0]

    def blocks():
        for r0 in range(0, bt, block_rows):
            r1 = min(bt, r0 + block_rows)
            yield r0, r1, z_s[r0:r1], z_t[r0:r1]

    return _from_logit_blocks(blocks(), x_s, w_s, labels, beta, temperature, reduction,
                              ignore_index, row_grad, False)


def _from_logit_blocks(blocks, x_s, w_s, labels, beta, temperature, reduction, ignore_index,
                       row_grad, emulate_rounding):
    bt, h_s = x_s.shape
    v = w_s.shape[0]
    w, valid, n = row_weights(labels, bt, v, reduction, ignore_index, row_grad)
    loss_rows = np.zeros(bt)
    grad_input = np.zeros((bt, h_s))
    grad_weight = np.zeros((v, h_s))
    for r0, r1, zs, zt in blocks:
        L, dA = jsd_rows(zs, zt, beta, temperature)
        vb = valid[r0:r1]
        L = np.where(vb, L, 0.0)
        loss_rows[r0:r1] = L
        dz = dA * (w[r0:r1] / temperature)[:, None]
        dz[~vb] = 0.0
        if emulate_rounding:
            dz = _store_round(dz, emulate_rounding)
        grad_input[r0:r1] = dz @ w_s
        grad_weight += dz.T @ x_s[r0:r1]
    if reduction == "none":
        loss = loss_rows
    elif n == 0:
        loss = 0.0
    elif reduction == "sum":
        loss = float(loss_rows.sum())
    elif reduction == "batchmean":
        loss = float(loss_rows.sum() / n)
    else:
        loss = float(loss_rows.sum() / (n * v))
    return loss, grad_input, grad_weight


def fljsd_rows_ref(x_s_rows, w_s, x_t_rows, w_t, *, beta: float, temperature: float,
                   row_scale):
    """Per-row loss L_r and grad_input rows for a sample of rows.

    Each row of the method is independent once its weight w_r is known
    (PR 1352, "Details": the kernel works row by row over V), so a sample of
    rows can be checked at any problem size. ``row_scale`` is w_r for each
    sampled row (for batchmean 1/n of the whole problem). Returns (L, dz,
    grad_input_rows).
    """
    zs = logits(x_s_rows, w_s)
    zt = logits(x_t_rows, w_t)
    L, dA = jsd_rows(zs, zt, beta, temperature)
    dz = dA * (np.asarray(row_scale, dtype=np.float64) / temperature)[:, None]
    return L, dz, dz @ np.asarray(w_s, dtype=np.float64)


# ---------------------------------------------------------------------------
# total variation distance (adjacent path; pins the batchmean reading)
# ---------------------------------------------------------------------------
def _dist_weights(labels, rows: int, v: int, reduction: str, ignore_index: int):
    """Row mask and per-row weight for the distances over given distributions
    (same reductions as the fused loss; none -> weight 1)."""
    w, valid, n = row_weights(labels, rows, v, "sum" if reduction == "none" else reduction,
                              ignore_index)
    return valid, n, w


def tvd_ref(p: np.ndarray, q: np.ndarray, reduction: str = "batchmean", labels=None,
            ignore_index: int = -100):
    """TVD loss 0.5*|p - q| summed over the vocabulary and its gradient in p.

    "Fix TVD gradient at p == q" (PR 1374), "Summary": the derivative of
    0.5*|p - q| is +0.5 where p > q, -0.5 where p < q, and exactly 0 at p == q
    (the three-way sign). Reductions follow the same readings as the JSD; the
    tie table of that page fixes batchmean as division by the number of rows.
    Rows whose label is ignore_index give loss 0 and gradient 0.
    Returns (loss, grad_p); loss is per element [rows x V] for none.
    """
    p = np.asarray(p, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    rows, v = p.shape
    if reduction not in REDUCTIONS:
        raise ValueError(reduction)
    valid, n, w = _dist_weights(labels, rows, v, reduction, ignore_index)
    per_elem = np.where(valid[:, None], 0.5 * np.abs(p - q), 0.0)
    sign = np.where(p > q, 1.0, np.where(p < q, -1.0, 0.0))
    grad = 0.5 * sign * w[:, None]
    if reduction == "none":
        return per_elem, grad
    total = per_elem.sum()
    if n == 0:
        return 0.0, grad
    scale = {"sum": 1.0, "batchmean": 1.0 / n, "mean": 1.0 / (n * v)}[reduction]
    return float(total * scale), grad


def dist_zero_masks(kind: str, x: np.ndarray, y: np.ndarray, *, beta: float = 0.5,
                    labels=None, ignore_index: int = -100):
    """Exact zeros of the two distances over given distributions, from the tie
    rule of PR 1374 "Summary" (x == y element by element) and the ignored rows.

    kind "tvd": the gradient 0.5 sign(p - q) is 0 at p == q, and the
    per-element loss 0.5 |p - q| is 0 there. kind "jsd" (log-space): the
    per-element loss is 0 at X == Y in every branch; the gradient is 0 there
    only in the generalized branch ((1 - beta) Q (X - log M), with M = Q);
    the endpoint gradients -P and Q (X - Y + 1) are not 0 at a tie.
    Returns (elem_loss_zero [rows x V], grad_zero [rows x V]); ignored rows are
    all True.
    """
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    tie = x == y
    rows = x.shape[0]
    valid = np.ones(rows, dtype=bool) if labels is None else \
        np.asarray(labels).reshape(-1) != ignore_index
    loss_zero = tie.copy()
    if kind == "tvd" or (0.0 < beta < 1.0):
        grad_zero = tie.copy()
    else:
        grad_zero = np.zeros_like(tie)
    loss_zero[~valid] = True
    grad_zero[~valid] = True
    return loss_zero, grad_zero


def jsd_logspace_ref(x: np.ndarray, y: np.ndarray, *, beta: float = 0.5,
                     reduction: str = "batchmean", labels=None, ignore_index: int = -100):
    """The generalized JSD on given log-probabilities and its gradient in X.

    The public contract of Liger's _jsd_kernel ("[Perf] Fuse log-softmax into
    fused_linear_jsd kernel", PR 1352, Open questions 3): the inputs are
    log-probabilities already, X = log Q (input, student) and Y = log P
    (target, teacher). Per element, with P = e^Y, Q = e^X and
    M = beta P + (1 - beta) Q: beta = 0 gives P (Y - X), beta = 1 gives
    Q (X - Y), otherwise beta P (Y - log M) + (1 - beta) Q (X - log M). The
    gradient is taken element by element with X as the free variable (the
    inputs are not renormalised): -P, Q (X - Y + 1), and (1 - beta) Q (X - log M).
    The tie rule of PR 1374 gives a zero loss term at X == Y, and a zero
    gradient where the calculus does (the generalized branch).
    Returns (loss, grad_x); loss is per row [rows] for none.
    """
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    rows, v = x.shape
    if not (0.0 <= beta <= 1.0):
        raise ValueError("beta must be in [0, 1]")
    valid, n, w = _dist_weights(labels, rows, v, reduction, ignore_index)
    P, Q = np.exp(y), np.exp(x)
    tie = x == y
    if beta == 0.0:
        ell = np.where(tie, 0.0, P * (y - x))
        g = -P
    elif beta == 1.0:
        ell = np.where(tie, 0.0, Q * (x - y))
        g = Q * (x - y + 1.0)
    else:
        M = beta * P + (1.0 - beta) * Q
        zero = tie | (M == 0.0)
        logM = np.log(np.where(M == 0.0, 1.0, M))
        ell = np.where(zero, 0.0, beta * P * (y - logM) + (1.0 - beta) * Q * (x - logM))
        g = np.where(zero, 0.0, (1.0 - beta) * Q * (x - logM))
    rows_loss = np.where(valid, ell.sum(axis=1), 0.0)
    grad = g * w[:, None]
    grad[~valid] = 0.0
    if reduction == "none":
        return rows_loss, grad
    if n == 0:
        return 0.0, grad
    scale = {"sum": 1.0, "batchmean": 1.0 / n, "mean": 1.0 / (n * v)}[reduction]
    return float(rows_loss.sum() * scale), grad


# ---------------------------------------------------------------------------
# fused linear cross-entropy (the FLCE path)
# ---------------------------------------------------------------------------
def flce_ref(x, w, labels, *, reduction: str = "mean", ignore_index: int = -100,
             label_smoothing: float = 0.0, lse_square_scale: float = 0.0, softcap: float = 0.0,
             block_rows: int = 256):
    """Cross-entropy of the logits x . w^T and its gradients in x and w.

    "perf(flce): write the weight-gradient product directly into grad_weight"
    (PR 1429): grad_weight is the sum over row chunks of dlogits^T . x; the
    page's tests exercise label smoothing, z-loss, softcap and reduction none.
    Per row with label y: c = softcap * tanh(z / softcap) (or z), lse =
    logsumexp(c), L = lse - (1 - eps) c_y - eps * mean_j(c_j) + lambda lse^2.
    Reductions: none -> per row; sum; mean (and batchmean) -> divided by the
    rows whose label is not ignore_index. Returns (loss, grad_input, grad_weight).
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    labels = np.asarray(labels).reshape(-1)
    bt, h = x.shape
    v = w.shape[0]
    valid = labels != ignore_index
    n = int(valid.sum())
    if reduction == "none" or reduction == "sum":
        scale = 1.0
    else:
        scale = 1.0 / n if n > 0 else 0.0
    eps, lam = label_smoothing, lse_square_scale
    loss_rows = np.zeros(bt)
    gi = np.zeros((bt, h))
    gw = np.zeros((v, h))
    for r0 in range(0, bt, block_rows):
        r1 = min(bt, r0 + block_rows)
        z = logits(x[r0:r1], w)
        c = softcap * np.tanh(z / softcap) if softcap > 0.0 else z
        m = c.max(axis=1, keepdims=True)
        lse = (m + np.log(np.exp(c - m).sum(axis=1, keepdims=True)))[:, 0]
        p = np.exp(c - lse[:, None])
        vb = valid[r0:r1]
        y = np.where(vb, labels[r0:r1], 0)
        cy = c[np.arange(r1 - r0), y]
        L = lse - (1.0 - eps) * cy - eps * c.mean(axis=1) + lam * lse ** 2
        loss_rows[r0:r1] = np.where(vb, L, 0.0)
        dc = p * (1.0 + 2.0 * lam * lse)[:, None] - eps / v
        dc[np.arange(r1 - r0), y] -= (1.0 - eps)
        if softcap > 0.0:
            dc = dc * (1.0 - (c / softcap) ** 2)
        dc[~vb] = 0.0
        dz = dc * scale
        gi[r0:r1] = dz @ w
        gw += dz.T @ x[r0:r1]
    if reduction == "none":
        return loss_rows, gi, gw
    return float(loss_rows.sum() * scale), gi, gw
