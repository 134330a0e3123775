"""GPU parity: the CUDA library against the float64 CPU oracle on the same seeded
inputs, element by element, with the stated tolerances (loss relative error
<= 1e-5 fp32 / 2e-3 bf16; gradient relative Frobenius error <= 1e-5 fp32 /
1e-2 bf16; exactly 0.0 wherever the oracle is exactly 0)."""
import numpy as np
import pytest
import torch

import jsd_inputs
import oracle
from parity_util import (TOL, assert_exact_zeros, compare, f64, method_zeros, oracle_zeros,
                         rel_fro, run_gpu, tile_errors)

pytestmark = pytest.mark.gpu

BETAS = (0.0, 0.1, 0.5, 1.0)
REDS = ("none", "sum", "mean", "batchmean")


def _oracle(inputs, **kw):
    x_s, w_s, x_t, w_t, labels = inputs
    return oracle.fljsd_ref(f64(x_s), f64(w_s), f64(x_t), f64(w_t), f64(labels), **kw)


# ---------------------------------------------------------------------------
# tiny fp32: every branch, temperature and reduction
# ---------------------------------------------------------------------------
@pytest.fixture(scope="module")
def tiny():
    return jsd_inputs.make_inputs(jsd_inputs.WORKLOADS["tiny_fp32"], "cpu")


@pytest.mark.parametrize("beta", BETAS)
@pytest.mark.parametrize("T", [1.0, 2.0])
@pytest.mark.parametrize("red", REDS)
def test_tiny_fp32(tiny, beta, T, red):
    out = run_gpu(*tiny, beta=beta, temperature=T, reduction=red)
    ref = _oracle(tiny, beta=beta, temperature=T, reduction=red)
    compare(out, ref, "fp32", f"tiny beta={beta} T={T} {red}",
            zeros=oracle_zeros(tiny, beta, T))
    for k, e in tile_errors(f64(out[2]), ref[2], 1000).items():
        assert e <= TOL["fp32"][1], (k, e)


# ---------------------------------------------------------------------------
# ties: self-distillation gives exact zeros; padded vocabulary
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("copies", [False, True])
@pytest.mark.parametrize("beta", BETAS)
def test_self_distillation_exact_zeros(beta, copies):
    w = jsd_inputs.WORKLOADS["ties_self"]
    x_s, w_s, x_t, w_t, labels = jsd_inputs.make_inputs(w, "cuda:0")
    if copies:
        x_t, w_t = x_s.clone(), w_s.clone()
    loss, gi, gw = run_gpu(x_s, w_s, x_t, w_t, labels, beta=beta, temperature=w.temperature,
                           reduction=w.reduction)
    assert loss.item() == 0.0
    assert int(torch.count_nonzero(gi)) == 0 and int(torch.count_nonzero(gw)) == 0


def test_padded_vocab():
    w = jsd_inputs.WORKLOADS["ties_padded"]
    inputs = jsd_inputs.make_inputs(w, "cpu")
    out = run_gpu(*inputs, beta=w.beta, temperature=w.temperature, reduction=w.reduction)
    ref = _oracle(inputs, beta=w.beta, temperature=w.temperature, reduction=w.reduction)
    compare(out, ref, "bf16", "padded vocab",
            zeros=oracle_zeros(inputs, w.beta, w.temperature))


# ---------------------------------------------------------------------------
# partially tied rows: the tie rule element by element
# ---------------------------------------------------------------------------
PARTIAL_CASES = {
    # name: (bt, h, v, dtype)
    "fp32_v1000": (64, 128, 1000, "fp32"),
    "bf16_v40960": (512, 256, 40960, "bf16"),
    "bf16_v33000": (384, 192, 33000, "bf16"),  # ragged last GEMM and pass-1 tiles
}


def _diff_cols(v):
    """Columns where student and teacher differ: tile edges of both the
    256-column GEMM tiles and the 128-column pass-1 partials, the last
    columns, and one inside."""
    return sorted({0, 127, 128, 255, 256, v // 2 + 3, v - 129, v - 128, v - 1})


@pytest.mark.parametrize("beta", BETAS)
@pytest.mark.parametrize("case", list(PARTIAL_CASES))
def test_partial_ties(case, beta):
    """Rows that tie at every column but a few (jsd_inputs.make_partial_ties),
    rows tied everywhere, rows tied nowhere, and ignored rows. The tie rule
    (PR 1374 "Summary"; carried to the logit gradient by PR 1352 "Details")
    fixes exact zeros that the oracle's tie mask locates: at beta = 0 every
    tied element's dlogit (Q - P)/T is exactly 0; rows tied everywhere and
    ignored rows are exactly 0 in every branch. The dlogits are read where the
    method leaves them, in place over the student logits in the workspace
    (one chunk). The tied elements of partially tied rows in the other
    branches (-Q L, -Q dX_sum: tiny but not 0) and the untied columns are
    compared with the oracle, as are the grad_weight rows at the kernels'
    tile edges and in the last vocabulary tile."""
    from lm_head_jsd_gb300 import FusedLinearJSD

    bt, h, v, dt = PARTIAL_CASES[case]
    tol_loss, tol_grad = TOL[dt]
    D = _diff_cols(v)
    for T in (1.0, 2.0):
        inputs, kinds = jsd_inputs.make_partial_ties(
            bt, h, v, dt, 91 + v % 97, temperature=T, diff_cols=D, n_full=bt // 16,
            n_free=bt // 8, ignore_frac=0.1)
        x_s, w_s, x_t, w_t, labels = (f64(t) for t in inputs)
        zs, zt = oracle.logits(x_s, w_s), oracle.logits(x_t, w_t)
        zeros = method_zeros(zs, zt, labels, beta, T)
        valid = labels != -100
        part = (kinds == "partial") & valid
        # the construction: partial rows tie off D and nowhere on D
        tie = oracle.tie_mask(zs, zt, T)
        off = np.ones(v, bool)
        off[D] = False
        assert np.all(tie[part][:, off]) and not np.any(tie[part][:, D])
        assert np.all(tie[kinds == "full"]) and not np.any(tie[kinds == "free"])

        dev_in = [t.cuda() for t in inputs]
        for red in ("batchmean", "none"):
            run = FusedLinearJSD(bt, h, h, v, inputs[0].dtype, beta=beta, temperature=T,
                                 reduction=red)
            assert run.plan.num_chunks == 1
            out = run.forward(*dev_in)
            torch.cuda.synchronize()
            what = f"{case} beta={beta} T={T} {red}"
            ref = oracle.fljsd_from_logits(zs, zt, x_s, w_s, labels, beta=beta, temperature=T,
                                           reduction=red)
            compare(out, ref, dt, what, zeros=zeros)
            # the dlogits, in place over the student logits (row stride ld)
            ld = run.plan.ld
            dz = f64(run.workspace[: bt * ld * inputs[0].element_size()]
                     .view(inputs[0].dtype).view(bt, ld)[:, :v])
            assert_exact_zeros(dz, zeros["dz"], what + " dlogits")
            if beta == 0.0:
                assert np.all(dz[part][:, off] == 0.0)  # tied elements of untied rows
            w_r, _, _ = oracle.row_weights(labels, bt, v, red)
            _, dA = oracle.jsd_rows(zs, zt, beta, T)
            dz_ref = dA * (w_r / T)[:, None]
            dz_ref[~valid] = 0.0
            e = rel_fro(dz[part][:, D], dz_ref[part][:, D])
            assert e <= tol_grad, f"{what}: dlogits at the untied columns {e:.3g}"
            if beta != 0.0:
                e = rel_fro(dz[part][:, off], dz_ref[part][:, off])
                assert e <= tol_grad, f"{what}: dlogits at tied columns {e:.3g}"
            for k, e in tile_errors(f64(out[2]), ref[2], v).items():
                assert e <= tol_grad, f"{what}: grad_weight {k} {e:.3g}"
            if beta == 0.0:
                # grad_input of a partially tied row draws only on the untied
                # columns, whose weight rows are 0 past hidden column 0
                gi = f64(out[1])
                assert np.all(gi[part][:, 1:] == 0.0)


# ---------------------------------------------------------------------------
# multi-block vocabulary with a partial trailing block: the full sweep
# ---------------------------------------------------------------------------
@pytest.fixture(scope="module")
def multiblock():
    w = jsd_inputs.WORKLOADS["multiblock"]
    inputs = jsd_inputs.make_inputs(w, "cpu")
    x_s, w_s, x_t, w_t, labels = (f64(t) for t in inputs)
    zs = oracle.logits(x_s, w_s)
    zt = oracle.logits(x_t, w_t)
    return inputs, (zs, zt, x_s, w_s, labels)


@pytest.mark.parametrize("beta", (0.0, 0.5, 1.0))
@pytest.mark.parametrize("T", (1.0, 2.0))
@pytest.mark.parametrize("red", REDS)
def test_multiblock_sweep(multiblock, beta, T, red):
    inputs, (zs, zt, x_s, w_s, labels) = multiblock
    out = run_gpu(*inputs, beta=beta, temperature=T, reduction=red)
    ref = oracle.fljsd_from_logits(zs, zt, x_s, w_s, labels, beta=beta, temperature=T,
                                   reduction=red)
    what = f"multiblock beta={beta} T={T} {red}"
    compare(out, ref, "bf16", what, zeros=method_zeros(zs, zt, labels, beta, T))
    for k, e in tile_errors(f64(out[2]), ref[2], zs.shape[1]).items():
        assert e <= TOL["bf16"][1], f"{what}: grad_weight {k} {e:.3g}"


# ---------------------------------------------------------------------------
# small and ragged shapes, chunking, upstream gradients
# ---------------------------------------------------------------------------
SMALL = [
    # (bt, h, v, dtype)
    (1, 8, 1, "bf16"), (1, 8, 7, "bf16"), (3, 16, 33, "bf16"), (130, 24, 1000, "bf16"),
    (257, 72, 4099, "bf16"), (1, 5, 1, "fp32"), (2, 7, 13, "fp32"), (65, 17, 1001, "fp32"),
    (129, 64, 9000, "bf16"),
    # H not a multiple of 8: the bf16 contractions run on the CUDA cores and
    # the row kernel forms pass 1 itself (no GEMM-epilogue partials)
    (33, 12, 1000, "bf16"), (70, 100, 2051, "bf16"),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("beta", (0.0, 0.3, 1.0))
def test_small_shapes(shape, beta):
    bt, h, v, dt = shape
    w = jsd_inputs.custom("small", 11 + bt + v, bt, h, v, dt, ignore_frac=0.25 if bt >= 4 else 0.0)
    inputs = jsd_inputs.make_inputs(w, "cpu")
    zeros = oracle_zeros(inputs, beta, 1.3)
    for red in ("none", "batchmean"):
        out = run_gpu(*inputs, beta=beta, temperature=1.3, reduction=red)
        ref = _oracle(inputs, beta=beta, temperature=1.3, reduction=red)
        compare(out, ref, dt, f"{shape} beta={beta} {red}", zeros=zeros)
        for k, e in tile_errors(f64(out[2]), ref[2], v).items():
            assert e <= TOL[dt][1], (shape, red, k, e)


@pytest.mark.parametrize("v", [122880, 131072])
def test_rows_longer_than_the_shared_cache(v):
    """bf16 rows of more than 114,688 columns: the row kernel's pass 3 takes
    X - log M of the first 114,688 from its shared-memory cache and recomputes
    the rest of the row from both logits. Every element against the oracle,
    tile edges included, and with the teacher equal to the student every
    gradient exactly 0."""
    w = jsd_inputs.custom("tmemrows", 61, 48, 64, v, "bf16", ignore_frac=0.1)
    inputs = jsd_inputs.make_inputs(w, "cpu")
    for red in ("batchmean", "none"):
        out = run_gpu(*inputs, beta=0.5, temperature=1.0, reduction=red)
        ref = _oracle(inputs, beta=0.5, temperature=1.0, reduction=red)
        compare(out, ref, "bf16", f"V={v} {red}", zeros=oracle_zeros(inputs, 0.5, 1.0))
        for k, e in tile_errors(f64(out[2]), ref[2], v).items():
            assert e <= TOL["bf16"][1], (v, red, k, e)
    x_s, w_s, _, _, labels = inputs
    loss, gi, gw = run_gpu(x_s, w_s, x_s, w_s, labels, beta=0.5, temperature=1.0)
    assert loss.item() == 0.0
    assert int(torch.count_nonzero(gi)) == 0 and int(torch.count_nonzero(gw)) == 0


@pytest.mark.parametrize("ignore_index", [7, 0])
def test_custom_ignore_index(ignore_index):
    """Rows whose label equals the given ignore_index (not -100) are skipped
    (loss 0, gradient rows exactly 0, n counts the rest); -100 is then an
    ordinary label whose rows count."""
    from lm_head_jsd_gb300 import FusedLinearJSD

    bt, h, v = 96, 64, 3000
    w = jsd_inputs.custom("ignidx", 51, bt, h, v, "bf16")
    x_s, w_s, x_t, w_t, _ = jsd_inputs.make_inputs(w, "cpu")
    labels = torch.randint(0, v, (bt,), generator=torch.Generator().manual_seed(52))
    labels[1::7] = -100
    labels[::5] = ignore_index
    for red in ("batchmean", "none"):
        run = FusedLinearJSD(bt, h, h, v, torch.bfloat16, beta=0.5, temperature=1.0,
                             reduction=red, ignore_index=ignore_index, device="cuda:0")
        out = run.forward(*(t.cuda() for t in (x_s, w_s, x_t, w_t, labels)))
        torch.cuda.synchronize()
        ref = oracle.fljsd_ref(f64(x_s), f64(w_s), f64(x_t), f64(w_t), labels.numpy(),
                               beta=0.5, temperature=1.0, reduction=red,
                               ignore_index=ignore_index)
        compare(out, ref, "bf16", f"ignore_index={ignore_index} {red}")
        ign = (labels == ignore_index).numpy()
        assert np.all(f64(out[1])[ign] == 0.0)
        if red == "none":
            assert np.all(f64(out[0])[ign] == 0.0) and np.all(f64(out[0])[~ign] != 0.0)


@pytest.mark.parametrize("chunk", [1, 7, 64, 128, 300])
def test_chunking_accumulates_grad_weight(chunk):
    w = jsd_inputs.custom("chunks", 21, 300, 64, 5000, "bf16", ignore_frac=0.1)
    inputs = jsd_inputs.make_inputs(w, "cpu")
    ref = _oracle(inputs, beta=0.5, temperature=1.0, reduction="batchmean")
    if chunk >= 64:
        # bf16 grad_weight is rounded once per chunk (PR 1429), so the bf16
        # tolerance holds for a handful of chunks, not for hundreds
        out = run_gpu(*inputs, beta=0.5, temperature=1.0, reduction="batchmean",
                      chunk_rows=chunk)
        compare(out, ref, "bf16", f"chunk={chunk}")
    out32 = run_gpu(*(t.float() if t is not None and t.is_floating_point() else t for t in inputs),
                    beta=0.5, reduction="batchmean", chunk_rows=chunk)
    compare(out32, ref, "fp32", f"fp32 chunk={chunk}")


def test_row_grad_with_reduction_none():
    w = jsd_inputs.custom("rowgrad", 31, 40, 32, 700, "fp32", ignore_frac=0.2)
    inputs = jsd_inputs.make_inputs(w, "cpu")
    rg = torch.linspace(-1.0, 2.0, 40)
    out = run_gpu(*inputs, beta=0.2, temperature=2.0, reduction="none", row_grad=rg)
    ref = _oracle(inputs, beta=0.2, temperature=2.0, reduction="none", row_grad=rg.numpy())
    compare(out, ref, "fp32", "row_grad")


def test_all_rows_ignored():
    w = jsd_inputs.custom("allign", 32, 16, 32, 300, "bf16")
    x_s, w_s, x_t, w_t, _ = jsd_inputs.make_inputs(w, "cpu")
    labels = torch.full((16,), -100, dtype=torch.int64)
    for red in REDS:
        loss, gi, gw = run_gpu(x_s, w_s, x_t, w_t, labels, reduction=red)
        assert torch.all(loss == 0) and torch.count_nonzero(gi) == 0
        assert torch.count_nonzero(gw) == 0


def test_backward_scales_by_grad_output():
    from lm_head_jsd_gb300 import FusedLinearJSD

    w = jsd_inputs.custom("bwd", 33, 64, 32, 500, "fp32")
    x_s, w_s, x_t, w_t, _ = (t.cuda() if t is not None else None
                             for t in jsd_inputs.make_inputs(w, "cpu"))
    run = FusedLinearJSD(64, 32, 32, 500, torch.float32)
    loss, gi, gw = run.forward(x_s, w_s, x_t, w_t)
    gi0, gw0 = gi.clone(), gw.clone()
    run.backward(torch.ones(1, device="cuda"), gi, gw)
    assert torch.equal(gi, gi0) and torch.equal(gw, gw0)
    run.backward(torch.full((1,), -2.5, device="cuda"), gi, gw)
    torch.testing.assert_close(gi, gi0 * -2.5, rtol=1e-6, atol=0)
    torch.testing.assert_close(gw, gw0 * -2.5, rtol=1e-6, atol=0)


def test_autograd_function():
    from lm_head_jsd_gb300 import fused_linear_jsd

    w = jsd_inputs.custom("autograd", 34, 48, 32, 600, "fp32", ignore_frac=0.1)
    x_s, w_s, x_t, w_t, labels = jsd_inputs.make_inputs(w, "cpu")
    xs = x_s.cuda().requires_grad_(True)
    ws = w_s.cuda().requires_grad_(True)
    loss = fused_linear_jsd(xs, ws, x_t.cuda(), w_t.cuda(), labels.cuda(), beta=0.4,
                            temperature=1.5, reduction="sum")
    (3.0 * loss).backward()
    ref = oracle.fljsd_ref(f64(x_s), f64(w_s), f64(x_t), f64(w_t), f64(labels), beta=0.4,
                           temperature=1.5, reduction="sum")
    assert abs(loss.item() - ref[0]) / abs(ref[0]) <= 1e-5
    assert rel_fro(f64(xs.grad), 3.0 * ref[1]) <= 1e-5
    assert rel_fro(f64(ws.grad), 3.0 * ref[2]) <= 1e-5
    # reduction="none" with a non-uniform upstream gradient
    xs.grad = None
    ws.grad = None
    rows = fused_linear_jsd(xs, ws, x_t.cuda(), w_t.cuda(), labels.cuda(), beta=0.4,
                            temperature=1.5, reduction="none")
    up = torch.linspace(0.5, 1.5, 48, device="cuda")
    (rows * up).sum().backward()
    ref = oracle.fljsd_ref(f64(x_s), f64(w_s), f64(x_t), f64(w_t), f64(labels), beta=0.4,
                           temperature=1.5, reduction="none", row_grad=f64(up))
    assert rel_fro(f64(xs.grad), ref[1]) <= 1e-5
    assert rel_fro(f64(ws.grad), ref[2]) <= 1e-5


def test_outputs_stay_inside_their_buffers():
    """Guard bands: outputs are views into larger buffers filled with a canary;
    nothing outside the views may change, and every element inside is written."""
    from lm_head_jsd_gb300 import FusedLinearJSD

    w = jsd_inputs.custom("guard", 35, 77, 40, 1234, "bf16", ignore_frac=0.1)
    x_s, w_s, x_t, w_t, labels = (t.cuda() for t in jsd_inputs.make_inputs(w, "cpu"))
    run = FusedLinearJSD(77, 40, 40, 1234, torch.bfloat16, reduction="none", chunk_rows=32)
    pad = 4096
    canary = 12345.0

    def guarded(n, dt):
        buf = torch.full((n + 2 * pad,), canary, dtype=dt, device="cuda")
        return buf, buf[pad:pad + n]

    lb, loss = guarded(77, torch.float32)
    gib, gi = guarded(77 * 40, torch.bfloat16)
    gwb, gw = guarded(1234 * 40, torch.bfloat16)
    run.forward(x_s, w_s, x_t, w_t, labels, out=(loss, gi.view(77, 40), gw.view(1234, 40)))
    torch.cuda.synchronize()
    for buf, n in ((lb, 77), (gib, 77 * 40), (gwb, 1234 * 40)):
        assert torch.all(buf[:pad] == canary) and torch.all(buf[pad + n:] == canary)
        assert not torch.any(buf[pad:pad + n] == canary)


def test_deterministic():
    w = jsd_inputs.custom("det", 36, 200, 64, 3000, "bf16", ignore_frac=0.1)
    inputs = jsd_inputs.make_inputs(w, "cpu")
    a = run_gpu(*inputs, beta=0.5)
    b = run_gpu(*inputs, beta=0.5)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("beta", BETAS)
@pytest.mark.parametrize("dt", ["fp32", "bf16"])
def test_extreme_temperature(beta, dt):
    """T = 0.02 multiplies the logits by 50. A group of 16 tokens leads both
    distributions (so they are not one-hot), while the other tokens' student and
    teacher log-probabilities differ by far more than 128 in log2 units: the
    ratio Q/P leaves the fp32 range and probabilities underflow, which must give
    finite, correct results.

    Tolerances: whatever error the logits carry is multiplied by 1/T in the
    scaled logits. In fp32 that is the GEMM's own accumulation error (about
    sqrt(K) ulps), so the fp32 tolerances are the stated T = 1 figures times
    1/T. In bf16 it is the storage rounding, so there the oracle rounds its
    logits and dlogits to bf16 as the kernels store them (its diagnostic mode)
    and the bf16 tolerances apply unchanged."""
    T = 0.02
    w = jsd_inputs.custom("extremeT", 51, 96, 64, 3000, dt, ignore_frac=0.1, spike=16)
    inputs = jsd_inputs.make_inputs(w, "cpu")
    for red in ("none", "sum"):
        out = run_gpu(*inputs, beta=beta, temperature=T, reduction=red)
        if dt == "fp32":
            ref = _oracle(inputs, beta=beta, temperature=T, reduction=red)
            compare(out, ref, dt, f"T={T} beta={beta} {dt} {red}", scale_tol=1.0 / T)
        else:
            ref = _oracle(inputs, beta=beta, temperature=T, reduction=red,
                          emulate_rounding="bf16")
            compare(out, ref, dt, f"T={T} beta={beta} {dt} {red}")


@pytest.mark.parametrize("beta", BETAS)
def test_saturated_rows(beta):
    """Independent student and teacher at T = 0.02: every row is one-hot at
    different tokens. For the KL endpoints the loss is large and the gradient
    (Q - P)/T is O(1/T): compared with the fp32 tolerances times 1/T (the fp32
    GEMM's error is magnified by 1/T). For the generalized JSD the loss sits at
    its bound h(beta) and the true gradient is about 1e-15 of the terms it is
    computed from -- below what any fp32 evaluation resolves (the float64
    oracle is at its own noise floor there): the loss must still match, and the
    gradients must be finite and tiny."""
    T = 0.02
    w = jsd_inputs.custom("saturated", 52, 96, 64, 3000, "fp32", ignore_frac=0.1)
    inputs = jsd_inputs.make_inputs(w, "cpu")
    out = run_gpu(*inputs, beta=beta, temperature=T, reduction="none")
    ref = _oracle(inputs, beta=beta, temperature=T, reduction="none")
    if beta in (0.0, 1.0):
        compare(out, ref, "fp32", f"saturated beta={beta}", scale_tol=1.0 / T)
        return
    loss, gi, gw = out
    assert rel_fro(f64(loss), ref[0]) <= 1e-5
    for g in (gi, gw):
        assert torch.all(torch.isfinite(g))
    # the terms are O(1/T) per element; fp32 leaves their difference near 1e-5
    assert float(gi.abs().max()) < 1e-2 and float(gw.abs().max()) < 1e-2


@pytest.mark.parametrize("dt", ["fp32", "bf16"])
@pytest.mark.parametrize("beta", (0.0, 0.5, 1.0))
def test_t2_scaling_flag(dt, beta):
    w = jsd_inputs.custom("t2", 61, 130, 64, 2000, dt, ignore_frac=0.1)
    inputs = jsd_inputs.make_inputs(w, "cpu")
    from lm_head_jsd_gb300 import FusedLinearJSD

    x_s, w_s, x_t, w_t, labels = (t.cuda() for t in inputs)
    for red in ("batchmean", "none"):
        run = FusedLinearJSD(130, 64, 64, 2000, w.torch_dtype, beta=beta, temperature=3.0,
                             reduction=red, t2_scale=True)
        out = run.forward(x_s, w_s, x_t, w_t, labels)
        torch.cuda.synchronize()
        ref = _oracle(inputs, beta=beta, temperature=3.0, reduction=red, t2_scale=True)
        compare(out, ref, dt, f"T^2 beta={beta} {red}")


@pytest.mark.parametrize("chunk", [1, 7, 64])
def test_fp32_grad_weight_accumulation(chunk, monkeypatch):
    """With the fp32 accumulator, hundreds of chunks stay within the bf16
    tolerance (without it, 300 one-row chunks drift to ~1.8e-2)."""
    from lm_head_jsd_gb300 import FusedLinearJSD

    w = jsd_inputs.custom("chunks", 21, 300, 64, 5000, "bf16", ignore_frac=0.1)
    inputs = jsd_inputs.make_inputs(w, "cpu")
    ref = _oracle(inputs, beta=0.5, temperature=1.0, reduction="batchmean")
    x_s, w_s, x_t, w_t, labels = (t.cuda() for t in inputs)
    run = FusedLinearJSD(300, 64, 64, 5000, torch.bfloat16, chunk_rows=chunk, accum_fp32=True)
    assert run.plan.workspace_bytes >= 5000 * 64 * 4
    out = [t.clone() for t in run.forward(x_s, w_s, x_t, w_t, labels)]
    torch.cuda.synchronize()
    compare(out, ref, "bf16", f"accum fp32 chunk={chunk}")
    # the accumulator read through TMA-prefetched slabs or through plain loads:
    # same arithmetic, same bits
    monkeypatch.setenv("FLJSD_GEMM_PREFETCH", "0")
    plain = run.forward(x_s, w_s, x_t, w_t, labels)
    torch.cuda.synchronize()
    for a, b in zip(out, plain):
        assert torch.equal(a, b)


@pytest.mark.parametrize("chunk", [1024, 384, 320])
@pytest.mark.parametrize("accum_fp32", [False, True], ids=["bf16_rmw", "fp32_acc"])
def test_chunked_grad_weight_on_cta_pairs(accum_fp32, chunk, monkeypatch):
    """Chunks of 1024, 384 or 320 rows make grad_weight a contraction deep
    enough for the CTA-pair schedule, so later chunks add into grad_weight (or
    the fp32 accumulator) through the pair kernel's read-modify-write epilogue
    (PR 1429 "Summary": first chunk overwrites, later chunks add and round
    once); at 384 and 320 rows the bf16 one runs two epilogue groups on a
    six-slab ring, and the last chunk is shorter. Against the oracle, and
    bitwise against one CTA per tile."""
    from lm_head_jsd_gb300 import FusedLinearJSD

    w = jsd_inputs.custom("pairchunks", 43, 3072, 64, 5000, "bf16", ignore_frac=0.1)
    inputs = jsd_inputs.make_inputs(w, "cpu")
    ref = _oracle(inputs, beta=0.5, temperature=1.0, reduction="batchmean")
    x_s, w_s, x_t, w_t, labels = (t.cuda() for t in inputs)
    outs = []
    for pair in ("1", "0"):
        monkeypatch.setenv("FLJSD_GEMM_PAIR", pair)
        run = FusedLinearJSD(3072, 64, 64, 5000, torch.bfloat16, chunk_rows=chunk,
                             accum_fp32=accum_fp32)
        assert run.plan.num_chunks == -(-3072 // chunk)
        outs.append([t.clone() for t in run.forward(x_s, w_s, x_t, w_t, labels)])
        torch.cuda.synchronize()
    compare(outs[0], ref, "bf16", f"pair chunks {chunk} accum_fp32={accum_fp32}",
            zeros=oracle_zeros(inputs, 0.5, 1.0))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("chunk", [128, 256])
def test_split_k_grad_input(chunk, monkeypatch):
    """A chunk with few output tiles splits the vocabulary contraction of
    grad_input; the fp32 partials are summed in a fixed order and rounded
    once. Loss and grad_weight do not depend on it (bitwise); grad_input
    differs from the unsplit contraction only by fp32 summation order."""
    w = jsd_inputs.custom("splitk", 41, 512, 512, 8192, "bf16", ignore_frac=0.1)
    inputs = jsd_inputs.make_inputs(w, "cpu")
    ref = _oracle(inputs, beta=0.5, temperature=1.0, reduction="batchmean")
    split = run_gpu(*inputs, beta=0.5, reduction="batchmean", chunk_rows=chunk)
    compare(split, ref, "bf16", f"split-K chunk={chunk}")
    again = run_gpu(*inputs, beta=0.5, reduction="batchmean", chunk_rows=chunk)
    for a, b in zip(split, again):
        assert torch.equal(a, b), "split-K result is not reproducible"
    monkeypatch.setenv("FLJSD_GEMM_SPLITK", "0")
    whole = run_gpu(*inputs, beta=0.5, reduction="batchmean", chunk_rows=chunk)
    compare(whole, ref, "bf16", f"unsplit chunk={chunk}")
    assert torch.equal(split[0], whole[0]) and torch.equal(split[2], whole[2])
    assert rel_fro(f64(split[1]), f64(whole[1])) <= 4e-3
