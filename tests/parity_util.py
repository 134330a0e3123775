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


def assert_exact_zeros(got, mask, what):
    """Every element (of a vector) or row (of a matrix) that ``mask`` marks as
    an exact zero of the method must be exactly 0.0."""
    got = np.asarray(got)
    mask = np.asarray(mask, dtype=bool)
    sel = got[mask]
    bad = int(np.count_nonzero(sel != 0.0))
    assert bad == 0, f"{what}: {bad} elements are nonzero where the method gives exactly 0"


def method_zeros(z_s, z_t, labels, beta, temperature):
    """The exact zeros of the method for rows with logits z_s, z_t, from the
    oracle's tie mask and the ignored rows (oracle.zero_masks): per-row losses
    that are 0, dlogits elements that are 0, and the grad_input rows and
    grad_weight (vocabulary) rows that are therefore sums of exact zeros."""
    import oracle

    loss_zero, dz_zero = oracle.zero_masks(z_s, z_t, labels, beta, temperature)
    return {"loss": loss_zero, "dz": dz_zero, "gi_rows": np.all(dz_zero, axis=1),
            "gw_rows": np.all(dz_zero, axis=0)}


def oracle_zeros(inputs, beta, temperature, block_rows=256):
    """method_zeros of a problem given by its inputs (logits formed by the
    oracle block by block)."""
    import oracle

    x_s, w_s, x_t, w_t, labels = (f64(t) for t in inputs)
    parts = []
    for r0 in range(0, x_s.shape[0], block_rows):
        r1 = min(x_s.shape[0], r0 + block_rows)
        zs = oracle.logits(x_s[r0:r1], w_s)
        zt = oracle.logits(x_t[r0:r1], w_t)
        parts.append(method_zeros(zs, zt, None if labels is None else labels[r0:r1], beta,
                                  temperature))
    return {"loss": np.concatenate([p["loss"] for p in parts]),
            "dz": np.concatenate([p["dz"] for p in parts]),
            "gi_rows": np.concatenate([p["gi_rows"] for p in parts]),
            "gw_rows": np.all(np.stack([p["gw_rows"] for p in parts]), axis=0)}


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


def compare(gpu, ref, dtype: str, what="", scale_tol: float = 1.0, zeros=None):
    """gpu = (loss, grad_input, grad_weight) tensors; ref = oracle outputs.
    ``zeros`` (from method_zeros / oracle_zeros) marks the method's exact
    zeros, which must come out as 0.0. ``scale_tol`` widens both tolerances
    (only for stress cases whose caller derives the factor from the
    arithmetic)."""
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
    if zeros is not None:
        if loss.size == zeros["loss"].size:  # reduction none: per-row losses
            assert_exact_zeros(loss, zeros["loss"], what + " loss rows")
        elif np.all(zeros["loss"]):
            assert np.all(loss == 0.0), f"{what}: every row is an exact zero, loss {loss}"
        assert_exact_zeros(gi, zeros["gi_rows"], what + " grad_input rows")
        assert_exact_zeros(gw, zeros["gw_rows"], what + " grad_weight rows")
    for name, g, r in (("grad_input", gi, rgi), ("grad_weight", gw, rgw)):
        assert np.all(np.isfinite(g)), f"{what}: {name} has non-finite values"
        if np.any(r != 0.0):
            e = rel_fro(g, r)
            assert e <= tol_grad, f"{what}: {name} rel Frobenius err {e:.3g} > {tol_grad}"
        else:
            assert np.all(g == 0.0), f"{what}: {name} nonzero where the oracle is all 0"


def tile_errors(got, ref, v):
    """Relative Frobenius errors of grad_weight on the vocabulary ranges where
    the kernels' tiling has edges: the last 256-column tile of the GEMMs (the
    partial one when V is not a multiple of 256) and the rows at every
    128-column boundary of the pass-1 partials (each side of the boundary).
    Returns {name: error}."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    last0 = (v - 1) // 256 * 256
    edges = sorted({j for b in range(128, v, 128) for j in (b - 1, b)})
    out = {"last_tile": rel_fro(got[last0:v], ref[last0:v])}
    if edges:
        out["stats_edges"] = rel_fro(got[edges], ref[edges])
    return out
