"""GPU parity of the fused linear cross-entropy against the float64 oracle:
options (label smoothing, z-loss, softcap, reductions, ignore_index), ragged
shapes, chunking with and without the fp32 grad_weight accumulator, invalid
labels, the autograd wrapper, and the full 8192 x 4096 x 128256 shape on
sampled rows."""
import itertools

import numpy as np
import pytest
import torch

import jsd_inputs
import oracle
from parity_util import TOL, compare, f64, rel_fro

pytestmark = pytest.mark.gpu


def _gpu(x, w, labels, dtype, chunk_rows=0, accum_fp32=False, **kw):
    from lm_head_jsd_gb300 import FusedLinearCrossEntropy

    dev = torch.device("cuda:0")
    run = FusedLinearCrossEntropy(x.shape[0], x.shape[1], w.shape[0],
                                  torch.float32 if dtype == "fp32" else torch.bfloat16,
                                  chunk_rows=chunk_rows, accum_fp32=accum_fp32, device=dev, **kw)
    out = run.forward(x.to(dev), w.to(dev), labels.to(dev))
    torch.cuda.synchronize()
    return out, run


OPTS = list(itertools.product(["mean", "sum", "none"], [0.0, 0.1], [0.0, 1e-3], [0.0, 15.0]))


@pytest.mark.parametrize("red,eps,lam,cap", OPTS)
def test_flce_tiny_fp32_options(red, eps, lam, cap):
    x, w, labels = jsd_inputs.make_ce_inputs(64, 128, 1000, "fp32", 101, ignore_frac=0.1)
    kw = dict(reduction=red, label_smoothing=eps, lse_square_scale=lam, softcap=cap)
    out, _ = _gpu(x, w, labels, "fp32", **kw)
    ref = oracle.flce_ref(f64(x), f64(w), labels.numpy(), **kw)
    compare(out, ref, "fp32", f"flce fp32 {kw}")


# (40, 12, 3001), (66, 100, 20003): H not a multiple of 8, so the bf16 GEMMs run
# on the CUDA cores and the row kernel forms pass 1 itself
@pytest.mark.parametrize("shape", [(1, 8, 7), (3, 16, 33), (130, 64, 4099), (257, 72, 32000),
                                   (40, 12, 3001), (66, 100, 20003)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("red", ["mean", "none"])
def test_flce_bf16_shapes(shape, red):
    bt, h, v = shape
    x, w, labels = jsd_inputs.make_ce_inputs(bt, h, v, "bf16", 102 + bt,
                                             ignore_frac=0.2 if bt >= 5 else 0.0)
    out, _ = _gpu(x, w, labels, "bf16", reduction=red, label_smoothing=0.05)
    ref = oracle.flce_ref(f64(x), f64(w), labels.numpy(), reduction=red, label_smoothing=0.05)
    compare(out, ref, "bf16", f"flce bf16 {shape} {red}")


# 256-row chunks: grad_weight contractions 256 deep run as CTA pairs
@pytest.mark.parametrize("chunk,acc", [(64, False), (128, False), (7, True), (1, True),
                                       (256, False), (256, True)])
def test_flce_chunking(chunk, acc):
    x, w, labels = jsd_inputs.make_ce_inputs(300, 64, 5000, "bf16", 103, ignore_frac=0.1)
    out, run = _gpu(x, w, labels, "bf16", chunk_rows=chunk, accum_fp32=acc)
    assert run.plan.num_chunks == -(-300 // chunk)
    ref = oracle.flce_ref(f64(x), f64(w), labels.numpy())
    compare(out, ref, "bf16", f"flce chunk={chunk} acc32={acc}")


# V = 20003 in bf16: 2500 vectors of 8 (the row kernel takes two per thread
# while v + 1024 < 2500, then one) and a ragged tail of 3 elements
LABEL_POSITIONS = ([0, 1, 2, 3, 4, 5, 6, 7]  # every lane of the first vector
                   + [8, 1023 * 8 + 7]  # the first vector's pair mate region
                   + [1024 * 8 + k for k in (0, 3, 7)]  # second vector of a pair
                   + [1475 * 8, 1476 * 8 + 5, 2048 * 8 + 3]  # last pair / one-at-a-time
                   + [2499 * 8, 2499 * 8 + 7]  # last full vector
                   + [20000, 20001, 20002])  # the tail


@pytest.mark.parametrize("eps,lam", [(0.0, 0.0), (0.1, 1e-3)])
def test_flce_label_positions(eps, lam):
    """The bf16 row kernel corrects the label's element once, by the thread
    whose vector holds it: labels on every lane of a vector, in both vectors
    of the two-deep loop, in the one-at-a-time remainder, in the last full
    vector and in the ragged tail; per-row losses and grad_input rows against
    the oracle, row by row."""
    v = 20003
    lab = torch.tensor(LABEL_POSITIONS + [-100, 12345], dtype=torch.int64)
    bt = lab.numel()
    x, w, _ = jsd_inputs.make_ce_inputs(bt, 64, v, "bf16", 107)
    kw = dict(label_smoothing=eps, lse_square_scale=lam)
    (loss, gi, gw), _ = _gpu(x, w, lab, "bf16", reduction="none", **kw)
    rows_ref, gi_ref, gw_ref = oracle.flce_ref(f64(x), f64(w), lab.numpy(), reduction="none",
                                               **kw)
    tol_loss, tol_grad = TOL["bf16"]
    got_l, got_gi = f64(loss), f64(gi)
    for r, y in enumerate(lab.tolist()):
        if y == -100:
            assert got_l[r] == 0.0 and np.all(got_gi[r] == 0.0), f"ignored row {r}"
            continue
        e = abs(got_l[r] - rows_ref[r]) / abs(rows_ref[r])
        assert e <= tol_loss, f"label {y}: loss {got_l[r]} vs {rows_ref[r]} ({e:.3g})"
        e = rel_fro(got_gi[r], gi_ref[r])
        assert e <= tol_grad, f"label {y}: grad_input row error {e:.3g}"
    assert rel_fro(f64(gw), gw_ref) <= tol_grad


@pytest.mark.parametrize("ignore_index", [5, 0])
def test_flce_custom_ignore_index(ignore_index):
    """A class id as ignore_index: rows with that label are skipped (loss 0,
    gradient rows exactly 0) and the mean divides by the other rows."""
    x, w, labels = jsd_inputs.make_ce_inputs(80, 64, 2500, "bf16", 108)
    labels[::4] = ignore_index
    for red in ("mean", "none"):
        out, _ = _gpu(x, w, labels, "bf16", reduction=red, ignore_index=ignore_index,
                      label_smoothing=0.1)
        ref = oracle.flce_ref(f64(x), f64(w), labels.numpy(), reduction=red,
                              ignore_index=ignore_index, label_smoothing=0.1)
        compare(out, ref, "bf16", f"flce ignore_index={ignore_index} {red}")
        ign = (labels == ignore_index).numpy()
        assert np.all(f64(out[1])[ign] == 0.0)


def test_flce_invalid_label_is_reported():
    from lm_head_jsd_gb300 import fljsd_workspace_status

    x, w, labels = jsd_inputs.make_ce_inputs(40, 32, 500, "fp32", 104)
    labels[5] = 500  # out of range
    (loss, gi, gw), run = _gpu(x, w, labels, "fp32", reduction="none")
    assert fljsd_workspace_status(run.plan, run.workspace) == 1
    assert loss[5].item() == 0.0 and int(torch.count_nonzero(gi[5])) == 0
    good = labels.clone()
    good[5] = -100
    ref = oracle.flce_ref(f64(x), f64(w), good.numpy(), reduction="none")
    compare((loss, gi, gw), ref, "fp32", "invalid label row skipped")


def test_flce_autograd():
    from lm_head_jsd_gb300 import fused_linear_cross_entropy

    x, w, labels = jsd_inputs.make_ce_inputs(48, 32, 700, "fp32", 105, ignore_frac=0.1)
    xt = x.cuda().requires_grad_(True)
    wt = w.cuda().requires_grad_(True)
    loss = fused_linear_cross_entropy(xt, wt, labels.cuda(), label_smoothing=0.1)
    (0.5 * loss).backward()
    ref = oracle.flce_ref(f64(x), f64(w), labels.numpy(), label_smoothing=0.1)
    assert abs(loss.item() - ref[0]) <= 1e-5 * abs(ref[0])
    assert rel_fro(f64(xt.grad), 0.5 * ref[1]) <= 1e-5
    assert rel_fro(f64(wt.grad), 0.5 * ref[2]) <= 1e-5


def test_flce_full_size_sampled_rows():
    """BT=8192, H=4096, V=128256 bf16, reduction mean (the benchmarked launch):
    sampled rows of grad_input and per-row losses against the oracle; then
    with only the sampled rows valid, the whole grad_weight."""
    bt, h, v = 8192, 4096, 128256
    dev = "cuda:0"
    x, w, labels = jsd_inputs.make_ce_inputs(bt, h, v, "bf16", 106, ignore_frac=0.05, device=dev)
    g = torch.Generator().manual_seed(7)
    R = torch.randperm(bt, generator=g)[:16].sort().values
    lab_np = labels.cpu().numpy()
    valid = lab_np != -100
    n = int(valid.sum())
    w64 = f64(w)
    xs = f64(x[R.to(dev)])
    rows_ref, gi_rows, _ = oracle.flce_ref(xs, w64, lab_np[R.numpy()], reduction="none")
    (loss, gi, gw), _ = _gpu(x, w, labels, "bf16", reduction="mean")
    assert rel_fro(f64(gi[R.to(dev)]), gi_rows / n) <= TOL["bf16"][1]
    del gi, gw
    (lrows, gi2, gw2), _ = _gpu(x, w, labels, "bf16", reduction="none")
    assert rel_fro(f64(lrows)[R.numpy()], rows_ref) <= TOL["bf16"][0]
    assert abs(loss.item() - f64(lrows).sum() / n) <= 1e-5 * abs(loss.item())
    del gi2, gw2
    torch.cuda.empty_cache()
    labC = torch.full((bt,), -100, dtype=torch.int64)
    labC[R] = labels.cpu()[R]
    (lC, giC, gwC), _ = _gpu(x, w, labC, "bf16", reduction="sum")
    _, _, gw_ref = oracle.flce_ref(xs, w64, labC.numpy()[R.numpy()], reduction="sum")
    assert rel_fro(f64(gwC), gw_ref) <= TOL["bf16"][1]
