"""Pins for the float64 CPU oracle: each test checks it against something other
than its own formulas -- library routines, textbook closed forms, brute force in
pure Python, finite differences, invariants of the mathematics, and the one
value the pages print (the TVD tie table)."""
import math
import os

import numpy as np
import pytest
import torch

from oracle import bf16_round, fljsd_ref, jsd_rows, row_weights, tvd_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
BETAS = (0.0, 0.1, 0.5, 1.0)


def _rng(seed):
    return np.random.default_rng(seed)


def _problem(seed, bt=4, h=8, v=16, h_t=None, scale=1.0):
    r = _rng(seed)
    h_t = h if h_t is None else h_t
    x_s = r.standard_normal((bt, h)) * scale
    w_s = r.standard_normal((v, h)) / math.sqrt(h)
    x_t = r.standard_normal((bt, h_t)) * scale
    w_t = r.standard_normal((v, h_t)) / math.sqrt(h_t)
    return x_s, w_s, x_t, w_t


# ---------------------------------------------------------------------------
# bf16 rounding helper
# ---------------------------------------------------------------------------
def test_bf16_round_known_values():
    # ulp(1) in bf16 is 2^-7; halfway cases round to the even neighbour.
    x = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, -2.5, 0.0,
                  3.0e38, 1e-40])
    got = bf16_round(x)
    assert got[0] == 1.0
    assert got[1] == 1.0                      # tie -> even (mantissa 0)
    assert got[2] == 1 + 2 ** -6              # tie -> even (mantissa 2)
    assert got[3] == 1 + 2 ** -7              # above half -> up
    assert got[4] == -2.5 and got[5] == 0.0


def test_bf16_round_matches_torch_conversion():
    x = _rng(0).standard_normal(100000) * np.exp(_rng(1).uniform(-20, 20, 100000))
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(bf16_round(x), ref)


# ---------------------------------------------------------------------------
# library routines and textbook forms at the endpoints
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1.0, 2.0])
def test_beta0_is_forward_kl_of_library(T):
    """beta=0 is KL(P||Q) with P the teacher: torch kl_div(input=log Q, target=log P)."""
    x_s, _, x_t, _ = _problem(3, bt=6, h=11, v=11)
    eye = np.eye(11)
    loss, _, _ = fljsd_ref(x_s, eye, x_t, eye, beta=0.0, temperature=T, reduction="batchmean")
    logq = torch.log_softmax(torch.from_numpy(x_s / T), dim=-1)
    logp = torch.log_softmax(torch.from_numpy(x_t / T), dim=-1)
    ref = torch.nn.functional.kl_div(logq, logp, log_target=True, reduction="batchmean").item()
    assert loss == pytest.approx(ref, rel=1e-12, abs=1e-15)


@pytest.mark.parametrize("T", [1.0, 3.0])
def test_beta1_is_reverse_kl_of_library(T):
    """beta=1 is KL(Q||P): torch kl_div(input=log P, target=log Q)."""
    x_s, _, x_t, _ = _problem(4, bt=5, h=9, v=9)
    eye = np.eye(9)
    loss, _, _ = fljsd_ref(x_s, eye, x_t, eye, beta=1.0, temperature=T, reduction="sum")
    logq = torch.log_softmax(torch.from_numpy(x_s / T), dim=-1)
    logp = torch.log_softmax(torch.from_numpy(x_t / T), dim=-1)
    ref = torch.nn.functional.kl_div(logp, logq, log_target=True, reduction="sum").item()
    assert loss == pytest.approx(ref, rel=1e-12)


@pytest.mark.parametrize("T", [1.0, 2.0])
def test_beta0_gradient_is_softmax_difference(T):
    """Soft-target cross-entropy gradient: d/dz_s = (softmax(z_s/T) - softmax(z_t/T)) / T."""
    from scipy.special import softmax

    x_s, _, x_t, _ = _problem(5, bt=7, h=13, v=13)
    eye = np.eye(13)  # logits == hidden states, so grad_input == dlogits
    _, gi, _ = fljsd_ref(x_s, eye, x_t, eye, beta=0.0, temperature=T, reduction="sum")
    ref = (softmax(x_s / T, axis=1) - softmax(x_t / T, axis=1)) / T
    np.testing.assert_allclose(gi, ref, rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------------------
# brute force in pure Python: the entropy form of the generalized JSD
# ---------------------------------------------------------------------------
def _py_softmax(row):
    m = max(row)
    e = [math.exp(x - m) for x in row]
    s = sum(e)
    return [x / s for x in e]


@pytest.mark.parametrize("beta", [0.1, 0.5, 0.9])
def test_generalized_matches_entropy_form(beta):
    """beta*KL(P||M) + (1-beta)*KL(Q||M) == H(M) - beta*H(P) - (1-beta)*H(Q),
    evaluated with plain Python loops (no NumPy) on a tiny case."""
    x_s, w_s, x_t, w_t = _problem(6, bt=3, h=5, v=7)
    T = 1.5
    loss_rows, _, _ = fljsd_ref(x_s, w_s, x_t, w_t, beta=beta, temperature=T, reduction="none")
    for r in range(3):
        zs = [sum(x_s[r][k] * w_s[j][k] for k in range(5)) / T for j in range(7)]
        zt = [sum(x_t[r][k] * w_t[j][k] for k in range(5)) / T for j in range(7)]
        q = _py_softmax(zs)
        p = _py_softmax(zt)
        m = [beta * pj + (1 - beta) * qj for pj, qj in zip(p, q)]

        def ent(d):
            return -sum(x * math.log(x) for x in d)

        ref = ent(m) - beta * ent(p) - (1 - beta) * ent(q)
        assert loss_rows[r] == pytest.approx(ref, rel=1e-10, abs=1e-14)


@pytest.mark.parametrize("T", [1.0, 2.0])
def test_beta_half_is_library_jensen_shannon(T):
    """At beta = 0.5 the generalized branch is the symmetric Jensen-Shannon
    divergence, whose square root scipy.spatial.distance.jensenshannon
    computes (natural log) from the two softmax distributions."""
    from scipy.spatial.distance import jensenshannon

    x_s, w_s, x_t, w_t = _problem(8, bt=5, h=16, v=300)
    loss_rows, _, _ = fljsd_ref(x_s, w_s, x_t, w_t, beta=0.5, temperature=T, reduction="none")
    zs = (x_s @ w_s.T) / T
    zt = (x_t @ w_t.T) / T
    q = np.exp(zs - zs.max(axis=1, keepdims=True))
    q /= q.sum(axis=1, keepdims=True)
    p = np.exp(zt - zt.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    for r in range(5):
        assert loss_rows[r] == pytest.approx(jensenshannon(p[r], q[r]) ** 2, rel=1e-9)


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("beta", BETAS)
@pytest.mark.parametrize("T", [1.0, 2.0])
@pytest.mark.parametrize("reduction", ["none", "sum", "mean", "batchmean"])
def test_identical_student_teacher_gives_exact_zeros(beta, T, reduction):
    x_s, w_s, _, _ = _problem(7, bt=6, h=12, v=40)
    loss, gi, gw = fljsd_ref(x_s, w_s, x_s.copy(), w_s.copy(), beta=beta, temperature=T,
                             reduction=reduction)
    assert np.all(np.asarray(loss) == 0.0)
    assert np.all(gi == 0.0) and np.all(gw == 0.0)


@pytest.mark.parametrize("beta", [0.1, 0.3, 0.5])
def test_beta_swap_symmetry(beta):
    """JSD_beta(P, Q) == JSD_{1-beta}(Q, P); at beta=0.5 the loss is symmetric."""
    r = _rng(8)
    zs, zt = r.standard_normal((9, 50)) * 3, r.standard_normal((9, 50)) * 3
    L1, _ = jsd_rows(zs, zt, beta, 1.0)
    L2, _ = jsd_rows(zt, zs, 1.0 - beta, 1.0)
    np.testing.assert_allclose(L1, L2, rtol=1e-12)


@pytest.mark.parametrize("beta", [0.1, 0.5, 0.9])
def test_bounds(beta):
    """0 <= L_r <= h(beta) = -beta ln beta - (1-beta) ln(1-beta) (<= ln 2 at 0.5)."""
    r = _rng(9)
    zs, zt = r.standard_normal((64, 30)) * 20, r.standard_normal((64, 30)) * 20
    L, _ = jsd_rows(zs, zt, beta, 1.0)
    hb = -beta * math.log(beta) - (1 - beta) * math.log(1 - beta)
    assert np.all(L >= 0.0) and np.all(L <= hb + 1e-12)
    if beta == 0.5:
        assert np.all(L <= math.log(2) + 1e-12)
    # far-apart one-hot-like distributions approach the bound
    zs1 = np.full((1, 4), -1e3); zs1[0, 0] = 0.0
    zt1 = np.full((1, 4), -1e3); zt1[0, 1] = 0.0
    L1, _ = jsd_rows(zs1, zt1, beta, 1.0)
    assert L1[0] == pytest.approx(hb, rel=1e-9)


def test_endpoint_limits():
    """JSD_beta / beta -> KL(P||Q) as beta -> 0; JSD_beta / (1-beta) -> KL(Q||P) as beta -> 1."""
    r = _rng(10)
    zs, zt = r.standard_normal((5, 60)), r.standard_normal((5, 60))
    eps = 1e-6
    L_lo, _ = jsd_rows(zs, zt, eps, 1.0)
    L_f, _ = jsd_rows(zs, zt, 0.0, 1.0)
    L_hi, _ = jsd_rows(zs, zt, 1.0 - eps, 1.0)
    L_r, _ = jsd_rows(zs, zt, 1.0, 1.0)
    np.testing.assert_allclose(L_lo / eps, L_f, rtol=2e-5)
    np.testing.assert_allclose(L_hi / eps, L_r, rtol=2e-5)
    # and the endpoint losses are the textbook KLs, computed here with scipy
    from scipy.special import rel_entr, softmax

    q, p = softmax(zs, axis=1), softmax(zt, axis=1)
    np.testing.assert_allclose(L_f, rel_entr(p, q).sum(axis=1), rtol=1e-11)
    np.testing.assert_allclose(L_r, rel_entr(q, p).sum(axis=1), rtol=1e-11)


@pytest.mark.parametrize("beta", BETAS)
def test_shift_invariance_and_zero_row_sum(beta):
    r = _rng(11)
    zs, zt = r.standard_normal((6, 33)) * 2, r.standard_normal((6, 33)) * 2
    L1, dA1 = jsd_rows(zs, zt, beta, 1.7)
    L2, dA2 = jsd_rows(zs + 5.25, zt - 3.5, beta, 1.7)
    np.testing.assert_allclose(L1, L2, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(dA1, dA2, rtol=1e-8, atol=1e-13)
    np.testing.assert_allclose(dA1.sum(axis=1), 0.0, atol=1e-14)


@pytest.mark.parametrize("beta", BETAS)
def test_temperature_rescaling(beta):
    """L(x; T) == L(x/T; 1) and grad_input(T) == grad_input_at_1(x/T) / T."""
    x_s, w_s, x_t, w_t = _problem(12, bt=5, h=6, v=20)
    T = 2.5
    l_t, gi_t, gw_t = fljsd_ref(x_s, w_s, x_t, w_t, beta=beta, temperature=T, reduction="sum")
    l_1, gi_1, gw_1 = fljsd_ref(x_s / T, w_s, x_t / T, w_t, beta=beta, temperature=1.0,
                                reduction="sum")
    assert l_t == pytest.approx(l_1, rel=1e-12)
    np.testing.assert_allclose(gi_t, gi_1 / T, rtol=1e-10, atol=1e-15)
    np.testing.assert_allclose(gw_t, gw_1, rtol=1e-10, atol=1e-15)


def test_ignored_rows_and_reductions():
    x_s, w_s, x_t, w_t = _problem(13, bt=8, h=6, v=25)
    labels = np.array([3, -100, 7, 0, -100, 24, 1, 2])
    n = 6
    out = {red: fljsd_ref(x_s, w_s, x_t, w_t, labels, beta=0.5, reduction=red)
           for red in ("none", "sum", "mean", "batchmean")}
    rows, gi_none, _ = out["none"]
    assert rows[1] == 0.0 and rows[4] == 0.0
    assert np.all(gi_none[1] == 0.0) and np.all(gi_none[4] == 0.0)
    assert out["sum"][0] == pytest.approx(rows.sum(), rel=1e-13)
    assert out["batchmean"][0] == pytest.approx(rows.sum() / n, rel=1e-13)
    assert out["mean"][0] == pytest.approx(rows.sum() / (n * 25), rel=1e-13)
    np.testing.assert_allclose(out["batchmean"][1] * n, out["sum"][1], rtol=1e-12)
    # the content of ignored rows does not matter
    x2 = x_s.copy(); x2[1] = 100.0
    l2, gi2, gw2 = fljsd_ref(x2, w_s, x_t, w_t, labels, beta=0.5, reduction="batchmean")
    assert l2 == out["batchmean"][0]
    np.testing.assert_array_equal(gw2, out["batchmean"][2])
    # every row ignored: zero loss and zero gradients, no NaN
    lz, giz, gwz = fljsd_ref(x_s, w_s, x_t, w_t, np.full(8, -100), reduction="batchmean")
    assert lz == 0.0 and np.all(giz == 0.0) and np.all(gwz == 0.0)


def test_row_blocking_does_not_change_the_result():
    x_s, w_s, x_t, w_t = _problem(14, bt=11, h=7, v=19)
    a = fljsd_ref(x_s, w_s, x_t, w_t, beta=0.1, temperature=2.0, block_rows=256)
    b = fljsd_ref(x_s, w_s, x_t, w_t, beta=0.1, temperature=2.0, block_rows=3)
    assert a[0] == pytest.approx(b[0], rel=1e-13)
    np.testing.assert_allclose(a[1], b[1], rtol=1e-12)
    np.testing.assert_allclose(a[2], b[2], rtol=1e-11, atol=1e-16)


# ---------------------------------------------------------------------------
# central finite differences
# ---------------------------------------------------------------------------
def _scalar_loss(x_s, w_s, x_t, w_t, labels, beta, T, red, row_grad):
    loss, _, _ = fljsd_ref(x_s, w_s, x_t, w_t, labels, beta=beta, temperature=T,
                           reduction=red, row_grad=row_grad)
    if red == "none":
        return float(np.sum(np.asarray(row_grad) * loss))
    return float(loss)


@pytest.mark.parametrize("beta", [0.0, 0.1, 0.5, 1.0])
@pytest.mark.parametrize("T", [1.0, 2.0])
@pytest.mark.parametrize("red", ["none", "sum", "mean", "batchmean"])
def test_finite_differences(beta, T, red):
    x_s, w_s, x_t, w_t = _problem(100 + int(beta * 10) + int(T), bt=4, h=8, v=16)
    labels = np.array([1, -100, 5, 2])
    row_grad = np.array([0.7, 1.3, -0.4, 2.0]) if red == "none" else None
    _, gi, gw = fljsd_ref(x_s, w_s, x_t, w_t, labels, beta=beta, temperature=T, reduction=red,
                          row_grad=row_grad)
    eps = 1e-6

    def fd(arr, idx, which):
        args = [x_s, w_s, x_t, w_t]
        plus = [a.copy() for a in args]; minus = [a.copy() for a in args]
        plus[which][idx] += eps; minus[which][idx] -= eps
        return (_scalar_loss(*plus, labels, beta, T, red, row_grad)
                - _scalar_loss(*minus, labels, beta, T, red, row_grad)) / (2 * eps)

    num_gi = np.array([[fd(x_s, (i, j), 0) for j in range(8)] for i in range(4)])
    num_gw = np.array([[fd(w_s, (i, j), 1) for j in range(8)] for i in range(16)])
    for num, ana in ((num_gi, gi), (num_gw, gw)):
        err = np.linalg.norm(num - ana) / max(np.linalg.norm(ana), 1e-30)
        assert err <= 1e-6, err
    assert np.all(gi[1] == 0.0)


@pytest.mark.parametrize("beta", BETAS)
def test_finite_differences_at_partial_ties(beta):
    """Rows where most columns tie (the teacher is the student with two logits
    swapped): the loss is smooth there, so finite differences give the true
    gradient, which the tie rule must not disturb."""
    r = _rng(15)
    v = 12
    x_s = r.standard_normal((3, v))
    x_t = x_s.copy()
    x_t[:, [2, 7]] = x_t[:, [7, 2]]
    eye = np.eye(v)
    _, gi, _ = fljsd_ref(x_s, eye, x_t, eye, beta=beta, temperature=1.0, reduction="sum")
    eps = 1e-6
    num = np.zeros_like(gi)
    for i in range(3):
        for j in range(v):
            p, m = x_s.copy(), x_s.copy()
            p[i, j] += eps; m[i, j] -= eps
            lp, _, _ = fljsd_ref(p, eye, x_t, eye, beta=beta, reduction="sum")
            lm, _, _ = fljsd_ref(m, eye, x_t, eye, beta=beta, reduction="sum")
            num[i, j] = (lp - lm) / (2 * eps)
    err = np.linalg.norm(num - gi) / np.linalg.norm(gi)
    assert err <= 1e-6, err


# ---------------------------------------------------------------------------
# the tie mask and the method's exact zeros
# ---------------------------------------------------------------------------
def _partial_tie_logits():
    """Row 0: the teacher equals the student except at column 3, where both
    logits sit 60 units below the row maximum (too small to move a float64
    sum of exponentials), so the log-normalisers are bitwise equal and every
    other column ties. Row 1: equal everywhere. Row 2: independent."""
    r = _rng(41)
    v = 10
    zs = r.standard_normal((3, v))
    zt = zs.copy()
    zs[0, 3] = zs[0].max() - 60.0
    zt[0, 3] = zs[0].max() - 58.0
    zt[2] = r.standard_normal(v)
    return zs, zt


def test_tie_mask_on_constructed_partial_ties():
    from oracle import tie_mask

    zs, zt = _partial_tie_logits()
    m = tie_mask(zs, zt, 1.0)
    expect = np.ones_like(m)
    expect[0, 3] = False
    expect[2] = False
    assert np.array_equal(m, expect)
    # a temperature that keeps column 3 far below the maximum keeps the ties
    assert np.array_equal(tie_mask(zs, zt, 1.5), expect)


@pytest.mark.parametrize("beta", BETAS)
def test_zero_masks_are_the_exact_zeros(beta):
    """The mask marks exactly the zeros the tie rule and ignored rows fix: the
    oracle's logit gradient is 0.0 there, and the tied elements of the
    partially tied row are left unmarked (and nonzero) outside beta = 0,
    where their gradient is -Q L (beta = 1) or -Q dX_sum."""
    from oracle import zero_masks

    zs, zt = _partial_tie_logits()
    labels = np.array([5, 1, 2, -100])
    zs = np.vstack([zs, zs[2]])
    zt = np.vstack([zt, zt[2]])
    loss_zero, dz_zero = zero_masks(zs, zt, labels, beta, 1.0)
    assert loss_zero.tolist() == [False, True, False, True]
    L, dA = jsd_rows(zs, zt, beta, 1.0)
    valid = labels != -100
    dA[~valid] = 0.0
    assert np.all(dA[dz_zero] == 0.0)
    assert np.all(L[1] == 0.0)
    tied_cols = np.ones(zs.shape[1], bool)
    tied_cols[3] = False
    assert np.all(dz_zero[1]) and np.all(dz_zero[3])
    if beta == 0.0:
        assert np.all(dz_zero[0, tied_cols]) and not dz_zero[0, 3]
    else:
        assert not np.any(dz_zero[0])
        assert np.all(dA[0, tied_cols] != 0.0)
    assert not np.any(dz_zero[2])


def test_dist_zero_masks():
    """TVD: the gradient is 0 exactly where p == q (PR 1374 "Summary"); the
    log-space JSD: every branch's loss term is 0 at a tie, the gradient only in
    the generalized branch (the endpoints' -P and Q (X - Y + 1) are not 0)."""
    from oracle import dist_zero_masks, jsd_logspace_ref

    r = _rng(43)
    p = r.random((3, 6)) + 0.1
    q = p.copy()
    q[0, [1, 4]] += 0.05
    q[2] = r.random(6) + 0.1
    labels = np.array([0, -100, 1])
    lz, gz = dist_zero_masks("tvd", p, q, labels=labels)
    ties = p == q
    assert np.array_equal(gz[[0, 2]], ties[[0, 2]]) and np.all(gz[1])
    _, g = tvd_ref(p, q, reduction="sum", labels=labels)
    assert np.all(g[gz] == 0.0) and np.all(g[~gz] != 0.0)
    x = np.log(p / p.sum(axis=1, keepdims=True))
    y = np.log(q / q.sum(axis=1, keepdims=True))
    y[0] = x[0]
    y[0, 2] -= 0.3
    for beta in BETAS:
        lz, gz = dist_zero_masks("jsd", x, y, beta=beta, labels=labels)
        _, g = jsd_logspace_ref(x, y, beta=beta, reduction="sum", labels=labels)
        assert np.all(g[gz] == 0.0)
        if beta in (0.0, 1.0):
            assert not np.any(gz[0]) and np.all(g[0] != 0.0)
        else:
            assert np.array_equal(gz[0], x[0] == y[0])


# ---------------------------------------------------------------------------
# the printed value: the TVD tie table pins batchmean = divide by rows
# ---------------------------------------------------------------------------
def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = v
    return vals


def test_tvd_tie_table():
    g = _golden("tvd_tie_batchmean.txt")
    rows, vocab = int(g["rows"]), int(g["vocab"])
    r = _rng(16)
    p = r.dirichlet(np.ones(vocab), size=rows).astype(np.float32).astype(np.float64)
    # p == q everywhere: every element is a tie and the gradient is exactly 0
    _, grad = tvd_ref(p, p.copy(), reduction=g["reduction"])
    assert np.all(grad == float(g["grad_at_tie_after_fix"]))
    assert int(np.sum(grad != 0.0)) == int(g["wrong_elements_after"])
    # the value a two-way split would have given at the tie (p < q branch)
    # is the p < q gradient: -0.5 / rows
    _, grad_lt = tvd_ref(p, p + 1e-3, reduction=g["reduction"])
    assert np.all(grad_lt == float(g["grad_at_tie_before_fix"]))
    assert int(np.sum(grad_lt != 0.0)) == int(g["wrong_elements_before"])


def test_row_weights_reading():
    w, valid, n = row_weights(np.array([1, -100, 2]), 3, 10, "mean")
    assert n == 2 and list(valid) == [True, False, True]
    np.testing.assert_allclose(w, [1 / 20, 0, 1 / 20])


def test_from_logits_matches_full_reference():
    from oracle import fljsd_from_logits, logits

    x_s, w_s, x_t, w_t = _problem(17, bt=9, h=5, v=21)
    labels = np.array([0, 1, -100, 3, 4, 5, -100, 7, 8])
    zs, zt = logits(x_s, w_s), logits(x_t, w_t)
    for red in ("none", "mean"):
        a = fljsd_ref(x_s, w_s, x_t, w_t, labels, beta=0.3, temperature=1.5, reduction=red)
        b = fljsd_from_logits(zs, zt, x_s, w_s, labels, beta=0.3, temperature=1.5, reduction=red,
                              block_rows=4)
        np.testing.assert_allclose(a[0], b[0], rtol=1e-13)
        np.testing.assert_allclose(a[1], b[1], rtol=1e-12)
        np.testing.assert_allclose(a[2], b[2], rtol=1e-11, atol=1e-16)


def test_rows_reference_matches_full_reference_rows():
    from oracle import fljsd_rows_ref

    x_s, w_s, x_t, w_t = _problem(18, bt=7, h=6, v=30)
    _, gi, _ = fljsd_ref(x_s, w_s, x_t, w_t, beta=0.2, temperature=1.7, reduction="sum")
    rows, _, _ = fljsd_ref(x_s, w_s, x_t, w_t, beta=0.2, temperature=1.7, reduction="none")
    idx = [1, 4, 6]
    L, dz, gir = fljsd_rows_ref(x_s[idx], w_s, x_t[idx], w_t, beta=0.2, temperature=1.7,
                                row_scale=np.ones(3))
    np.testing.assert_allclose(L, rows[idx], rtol=1e-13)
    np.testing.assert_allclose(gir, gi[idx], rtol=1e-12)


def test_storage_rounding_modes():
    """The diagnostic rounding: fp32 mode equals NumPy's float32 cast of the
    logits; bf16 mode equals the bf16 rounding pinned above."""
    from oracle import logits

    x_s, w_s, x_t, w_t = _problem(19, bt=5, h=6, v=40)
    for mode, rnd in (("fp32", lambda z: z.astype(np.float32).astype(np.float64)),
                      ("bf16", bf16_round)):
        got = fljsd_ref(x_s, w_s, x_t, w_t, beta=0.3, temperature=0.5, reduction="sum",
                        emulate_rounding=mode)
        from oracle import fljsd_from_logits

        ref = fljsd_from_logits(rnd(logits(x_s, w_s)), rnd(logits(x_t, w_t)), x_s, w_s, beta=0.3,
                                temperature=0.5, reduction="sum")
        assert got[0] == pytest.approx(ref[0], rel=1e-12)
        # dlogits are rounded in the mode too, so the gradients differ slightly
        assert np.linalg.norm(got[1] - ref[1]) <= 1e-2 * np.linalg.norm(ref[1])


def test_t2_scaling_reaches_the_high_temperature_limit():
    """Hinton et al. 2015, section 2.1: at high temperature the soft-target
    gradient (Q - P)/T approaches (z_s - z_t)/(N T^2) for zero-mean logits, so
    the T^2-scaled gradient approaches (z_s - z_t)/N, independent of T."""
    r = _rng(20)
    v = 17
    zs = r.standard_normal((3, v)); zs -= zs.mean(axis=1, keepdims=True)
    zt = r.standard_normal((3, v)); zt -= zt.mean(axis=1, keepdims=True)
    eye = np.eye(v)
    T = 1e4
    _, gi, _ = fljsd_ref(zs, eye, zt, eye, beta=0.0, temperature=T, reduction="sum",
                         t2_scale=True)
    ref = (zs - zt) / v
    # the next term of the expansion is O(|z| / T) relative
    assert np.linalg.norm(gi - ref) <= 1e-3 * np.linalg.norm(ref)
    loss1, gi1, gw1 = fljsd_ref(zs, eye, zt, eye, beta=0.3, temperature=2.0, reduction="sum")
    loss2, gi2, gw2 = fljsd_ref(zs, eye, zt, eye, beta=0.3, temperature=2.0, reduction="sum",
                                t2_scale=True)
    assert loss2 == pytest.approx(4.0 * loss1, rel=1e-14)
    np.testing.assert_allclose(gi2, 4.0 * gi1, rtol=1e-14)



# ---------------------------------------------------------------------------
# distances over given distributions
# ---------------------------------------------------------------------------
def _logprobs(seed, rows=5, v=23, scale=2.0):
    r = _rng(seed)
    a = r.standard_normal((rows, v)) * scale
    b = r.standard_normal((rows, v)) * scale
    lp = lambda z: z - np.log(np.exp(z - z.max(1, keepdims=True)).sum(1, keepdims=True)) \
        - z.max(1, keepdims=True)  # noqa: E731
    return lp(a), lp(b)


def test_logspace_endpoints_are_library_kl_with_autograd_gradients():
    from oracle import jsd_logspace_ref

    X, Y = _logprobs(30)
    for beta, inp, tgt in ((0.0, X, Y), (1.0, Y, X)):
        loss, grad = jsd_logspace_ref(X, Y, beta=beta, reduction="sum")
        xt = torch.tensor(X, requires_grad=True)
        yt = torch.tensor(Y)
        a, b = (xt, yt) if beta == 0.0 else (yt, xt)
        ref = torch.nn.functional.kl_div(a, b, log_target=True, reduction="sum")
        ref.backward()
        assert loss == pytest.approx(ref.item(), rel=1e-12)
        np.testing.assert_allclose(grad, xt.grad.numpy(), rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("beta", [0.1, 0.5, 0.8])
def test_logspace_generalized_matches_entropy_form_and_finite_differences(beta):
    from oracle import jsd_logspace_ref

    X, Y = _logprobs(31)
    rows, _ = jsd_logspace_ref(X, Y, beta=beta, reduction="none")
    for r in range(X.shape[0]):
        q = [math.exp(t) for t in X[r]]
        p = [math.exp(t) for t in Y[r]]
        m = [beta * a + (1 - beta) * b for a, b in zip(p, q)]
        ent = lambda d: -sum(t * math.log(t) for t in d)  # noqa: E731
        assert rows[r] == pytest.approx(ent(m) - beta * ent(p) - (1 - beta) * ent(q), rel=1e-10)
    # gradient in X as free variables
    _, grad = jsd_logspace_ref(X, Y, beta=beta, reduction="batchmean")
    eps = 1e-6
    num = np.zeros_like(X)
    for i in range(X.shape[0]):
        for j in range(X.shape[1]):
            a, b = X.copy(), X.copy()
            a[i, j] += eps; b[i, j] -= eps
            num[i, j] = (jsd_logspace_ref(a, Y, beta=beta)[0] - jsd_logspace_ref(b, Y, beta=beta)[0]) / (2 * eps)
    assert np.linalg.norm(num - grad) <= 1e-6 * np.linalg.norm(grad)


def test_logspace_ties_ignored_rows_and_reductions():
    from oracle import jsd_logspace_ref

    X, Y = _logprobs(32, rows=6)
    Y[2] = X[2]  # a fully tied row
    labels = np.array([0, -100, 3, 4, 5, 6])
    rows, g = jsd_logspace_ref(X, Y, beta=0.5, reduction="none", labels=labels)
    assert rows[2] == 0.0 and np.all(g[2] == 0.0)
    assert rows[1] == 0.0 and np.all(g[1] == 0.0)
    s, _ = jsd_logspace_ref(X, Y, beta=0.5, reduction="sum", labels=labels)
    b, _ = jsd_logspace_ref(X, Y, beta=0.5, reduction="batchmean", labels=labels)
    m, _ = jsd_logspace_ref(X, Y, beta=0.5, reduction="mean", labels=labels)
    assert s == pytest.approx(rows.sum()) and b == pytest.approx(s / 5)
    assert m == pytest.approx(s / (5 * X.shape[1]))


def test_tvd_matches_library_l1_and_autograd_off_ties():
    r = _rng(33)
    p = r.dirichlet(np.ones(40), size=6)
    q = r.dirichlet(np.ones(40), size=6)
    loss, grad = tvd_ref(p, q, reduction="sum")
    pt = torch.tensor(p, requires_grad=True)
    ref = 0.5 * torch.nn.functional.l1_loss(pt, torch.tensor(q), reduction="sum")
    ref.backward()
    assert loss == pytest.approx(ref.item(), rel=1e-13)
    np.testing.assert_allclose(grad, pt.grad.numpy(), rtol=0, atol=0)
    labels = np.array([1, -100, 2, 3, -100, 5])
    lb, gb = tvd_ref(p, q, reduction="batchmean", labels=labels)
    valid = labels != -100
    assert lb == pytest.approx(0.5 * np.abs(p - q)[valid].sum() / 4)
    assert np.all(gb[~valid] == 0.0)


# ---------------------------------------------------------------------------
# fused linear cross-entropy
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("eps", [0.0, 0.1])
@pytest.mark.parametrize("red", ["mean", "sum", "none"])
def test_flce_loss_is_library_cross_entropy(eps, red):
    from oracle import flce_ref

    x_s, w_s, _, _ = _problem(40, bt=9, h=6, v=30)
    labels = np.array([3, -100, 0, 29, 7, 7, -100, 1, 12])
    loss, gi, gw = flce_ref(x_s, w_s, labels, reduction=red, label_smoothing=eps)
    xt = torch.tensor(x_s, requires_grad=True)
    wt = torch.tensor(w_s, requires_grad=True)
    ref = torch.nn.functional.cross_entropy(xt @ wt.T, torch.tensor(labels), ignore_index=-100,
                                            label_smoothing=eps, reduction=red)
    if red == "none":
        np.testing.assert_allclose(loss, ref.detach().numpy(), rtol=1e-12, atol=1e-14)
        ref = ref.sum()
    else:
        assert loss == pytest.approx(ref.item(), rel=1e-12)
    ref.backward()
    np.testing.assert_allclose(gi, xt.grad.numpy(), rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(gw, wt.grad.numpy(), rtol=1e-10, atol=1e-14)


def test_flce_softcap_and_z_loss_gradients_match_autograd():
    from oracle import flce_ref

    x_s, w_s, _, _ = _problem(41, bt=7, h=5, v=20, scale=3.0)
    labels = np.array([0, 5, -100, 19, 3, 3, 8])
    cap, lam, eps = 2.5, 1e-3, 0.05
    loss, gi, gw = flce_ref(x_s, w_s, labels, reduction="mean", label_smoothing=eps,
                            lse_square_scale=lam, softcap=cap)
    xt = torch.tensor(x_s, requires_grad=True)
    wt = torch.tensor(w_s, requires_grad=True)
    c = cap * torch.tanh((xt @ wt.T) / cap)
    lab = torch.tensor(labels)
    valid = lab != -100
    lse = torch.logsumexp(c, dim=1)
    ce = torch.nn.functional.cross_entropy(c, lab, ignore_index=-100, label_smoothing=eps,
                                           reduction="sum")
    ref = (ce + lam * (lse[valid] ** 2).sum()) / valid.sum()
    ref.backward()
    assert loss == pytest.approx(ref.item(), rel=1e-12)
    np.testing.assert_allclose(gi, xt.grad.numpy(), rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(gw, wt.grad.numpy(), rtol=1e-10, atol=1e-14)
