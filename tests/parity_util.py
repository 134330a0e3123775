"""Helpers shared by the GPU parity tests: run the CUDA library, run the oracle
on the same tensors, and compare with the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

# loss relative error, gradient relative Frobenius error
TOL = {"fp32": (1e-5, 1e-5), "bf16": (2e-3, 1e-2)}


def f64(t):
    if t is None:
        return None
    return t.detach().to("cpu").to(torch.float64).numpy() if t.is_floating_point() else \
        t.detach().to("cpu").numpy()


def rel_fro(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    if den == 0.0:
        return float(np.linalg.norm(got))
    return float(np.linalg.norm(got - ref) / den)


def assert_zeros_where_ref_zero(got, ref, what):
    """Exact zeros of the method -- ignored rows, fully tied rows, an all-zero
    result -- must come out as exact zeros. They show as oracle rows (of a
    vector: elements) that are entirely 0.0; an isolated 0.0 inside a nonzero
    row is a numerical cancellation, not a zero of the method."""
    got = np.asarray(got)
    ref = np.asarray(ref)
    if ref.ndim == 1:
        mask = ref == 0.0
        bad = int(np.count_nonzero(got[mask] != 0.0))
    else:
        zero_rows = np.all(ref == 0.0, axis=1)
        bad = int(np.count_nonzero(got[zero_rows] != 0.0))
    assert bad == 0, f"{what}: {bad} elements are nonzero where the oracle is exactly 0"


def run_gpu(x_s, w_s, x_t, w_t, labels=None, *, beta=0.5, temperature=1.0,
            reduction="batchmean", chunk_rows=0, row_grad=None, device="cuda:0"):
    from lm_head_jsd_gb300 import FusedLinearJSD

    dev = torch.device(device)
    run = FusedLinearJSD(x_s.shape[0], x_s.shape[1], x_t.shape[1], w_s.shape[0], x_s.dtype,
                         beta=beta, temperature=temperature, reduction=reduction,
                         chunk_rows=chunk_rows, device=dev)
    mv = lambda t: None if t is None else t.to(dev).contiguous()  # noqa: E731
    loss, gi, gw = run.forward(mv(x_s), mv(w_s), mv(x_t), mv(w_t), mv(labels), mv(row_grad))
    torch.cuda.synchronize()
    return loss, gi, gw


def compare(gpu, ref, dtype: str, what="", scale_tol: float = 1.0):
    """gpu = (loss, grad_input, grad_weight) tensors; ref = oracle outputs.
    ``scale_tol`` widens both tolerances (only for stress cases whose caller
    derives the factor from the arithmetic)."""
    tol_loss, tol_grad = (t * scale_tol for t in TOL[dtype])
    loss, gi, gw = (f64(t) for t in gpu)
    rl, rgi, rgw = ref
    rl = np.atleast_1d(np.asarray(rl, dtype=np.float64))
    loss = loss.reshape(rl.shape)
    if np.all(rl == 0.0):
        assert np.all(loss == 0.0), f"{what}: loss {loss[:4]} where the oracle is exactly 0"
    else:
        e = rel_fro(loss, rl)
        assert e <= tol_loss, f"{what}: loss rel err {e:.3g} > {tol_loss}"
    assert_zeros_where_ref_zero(loss, rl, what + " loss")
    for name, g, r in (("grad_input", gi, rgi), ("grad_weight", gw, rgw)):
        assert np.all(np.isfinite(g)), f"{what}: {name} has non-finite values"
        assert_zeros_where_ref_zero(g, r, f"{what} {name}")
        if np.any(r != 0.0):
            e = rel_fro(g, r)
            assert e <= tol_grad, f"{what}: {name} rel Frobenius err {e:.3g} > {tol_grad}"
