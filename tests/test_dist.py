"""GPU parity of the distances over given distributions -- the log-space JSD
(Liger's _jsd_kernel contract) and TVD with the tie fix -- against the float64
oracle, with the same tolerances as the fused loss."""
import numpy as np
import pytest
import torch

import jsd_inputs
import oracle
from parity_util import TOL, assert_exact_zeros, f64, rel_fro

pytestmark = pytest.mark.gpu

SHAPES = [(1, 1), (3, 7), (64, 1000), (130, 4099), (257, 32000)]


def _run(kind, a, b, labels, dtype, reduction, beta=0.5):
    from lm_head_jsd_gb300 import _lib

    rows, v = a.shape
    dev = "cuda:0"
    a, b = a.to(dev), b.to(dev)
    lab = None if labels is None else labels.to(dev)
    loss = torch.empty((rows, v) if (kind == "tvd" and reduction == "none") else
                       ((rows,) if reduction == "none" else (1,)), dtype=torch.float32,
                       device=dev)
    grad = torch.empty_like(a)
    ws = torch.empty(_lib.fljsd_rows_workspace_bytes(rows), dtype=torch.uint8, device=dev)
    if kind == "tvd":
        _lib.fljsd_tvd(rows, v, dtype, reduction, -100, a, b, lab, loss, grad, ws)
    else:
        _lib.fljsd_jsd_logspace(rows, v, dtype, beta, reduction, -100, a, b, lab, loss, grad, ws)
    torch.cuda.synchronize()
    return loss, grad


def _check(loss, grad, ref, dtype, what, zeros):
    """Tolerances as for the fused loss; ``zeros`` = oracle.dist_zero_masks:
    where the method gives exact zeros (ties, ignored rows) the kernel must
    give 0.0 -- per element for the gradient and for TVD's per-element loss,
    per row (rows tied everywhere or ignored) for a per-row loss."""
    tol_loss, tol_grad = TOL[dtype]
    rl = np.atleast_1d(np.asarray(ref[0], dtype=np.float64))
    gl = f64(loss).reshape(rl.shape)
    if np.any(rl != 0.0):
        assert rel_fro(gl, rl) <= tol_loss, (what, rel_fro(gl, rl))
    else:
        assert np.all(gl == 0.0), what
    elem_zero, grad_zero = zeros
    if gl.shape == elem_zero.shape:
        assert_exact_zeros(gl, elem_zero, what + " loss")
    elif gl.shape == elem_zero.shape[:1]:
        assert_exact_zeros(gl, np.all(elem_zero, axis=1), what + " loss rows")
    gg = f64(grad)
    assert np.all(np.isfinite(gg))
    assert_exact_zeros(gg, grad_zero, what + " grad")
    if np.any(ref[1] != 0.0):
        assert rel_fro(gg, ref[1]) <= tol_grad, (what, rel_fro(gg, ref[1]))


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("beta", [0.0, 0.1, 0.5, 1.0])
def test_jsd_logspace(shape, dtype, beta):
    rows, v = shape
    a, b, labels = jsd_inputs.make_distributions(rows, v, dtype, 70 + rows, logspace=True,
                                                 tied_rows=1 if rows > 2 else 0,
                                                 tied_frac=0.1,
                                                 ignore_frac=0.1 if rows >= 10 else 0.0)
    for red in ("none", "sum", "mean", "batchmean"):
        loss, grad = _run("jsd", a, b, labels, dtype, red, beta)
        lab = None if labels is None else labels.numpy()
        ref = oracle.jsd_logspace_ref(f64(a), f64(b), beta=beta, reduction=red, labels=lab)
        zeros = oracle.dist_zero_masks("jsd", f64(a), f64(b), beta=beta, labels=lab)
        _check(loss, grad, ref, dtype, f"jsd {shape} {dtype} beta={beta} {red}", zeros)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_tvd(shape, dtype):
    rows, v = shape
    a, b, labels = jsd_inputs.make_distributions(rows, v, dtype, 80 + rows, logspace=False,
                                                 tied_rows=1 if rows > 2 else 0,
                                                 tied_frac=0.25,
                                                 ignore_frac=0.1 if rows >= 10 else 0.0)
    for red in ("none", "sum", "mean", "batchmean"):
        loss, grad = _run("tvd", a, b, labels, dtype, red)
        lab = None if labels is None else labels.numpy()
        ref = oracle.tvd_ref(f64(a), f64(b), reduction=red, labels=lab)
        zeros = oracle.dist_zero_masks("tvd", f64(a), f64(b), labels=lab)
        _check(loss, grad, ref, dtype, f"tvd {shape} {dtype} {red}", zeros)
        # the gradient is exactly +-0.5 w or 0: compare it exactly
        assert np.array_equal(f64(grad), ref[1].astype(np.float32).astype(
            np.float64) if dtype == "fp32" else f64(torch.from_numpy(ref[1]).to(torch.bfloat16)))


def test_tvd_tie_table_on_gpu():
    """The printed case: (8, 512) fp32, p == q everywhere, batchmean: the
    gradient is 0.0 at every element (and -0.0625 on the p < q side)."""
    p = torch.softmax(torch.randn(8, 512, generator=torch.Generator().manual_seed(9)), -1)
    loss, grad = _run("tvd", p, p.clone(), None, "fp32", "batchmean")
    assert loss.item() == 0.0 and int(torch.count_nonzero(grad)) == 0
    loss, grad = _run("tvd", p, p + 1e-3, None, "fp32", "batchmean")
    assert torch.all(grad == -0.0625)


def test_autograd_wrappers():
    from lm_head_jsd_gb300 import jsd_logspace, tvd

    a, b, _ = jsd_inputs.make_distributions(16, 300, "fp32", 90, logspace=True)
    x = a.cuda().requires_grad_(True)
    loss = jsd_logspace(x, b.cuda(), beta=0.3, reduction="sum")
    (2.0 * loss).backward()
    ref = oracle.jsd_logspace_ref(f64(a), f64(b), beta=0.3, reduction="sum")
    assert abs(loss.item() - ref[0]) <= 1e-5 * abs(ref[0])
    assert rel_fro(f64(x.grad), 2.0 * ref[1]) <= 1e-5
    p, q, _ = jsd_inputs.make_distributions(16, 300, "fp32", 91, logspace=False)
    pt = p.cuda().requires_grad_(True)
    l2 = tvd(pt, q.cuda(), reduction="batchmean")
    l2.backward()
    ref = oracle.tvd_ref(f64(p), f64(q), reduction="batchmean")
    assert abs(l2.item() - ref[0]) <= 1e-5 * abs(ref[0])
    assert rel_fro(f64(pt.grad), ref[1]) <= 1e-6
