"""fljsd_forward_noalloc, the forward for callers that cannot allocate device
memory -- a plugin running inside a host framework that owns every device
allocation and hands over only the input and output buffers has no way to
obtain the workspace fljsd_forward needs, so this entry point takes its scratch
from a fixed array inside the library instead.

Checked through the C ABI against fljsd_forward with a caller-provided
workspace, with the tolerances of the parity tests, on two calls in a row with
different problems (the second call runs over whatever the first left in the
shared array). Kept in a file that pytest collects last.
"""
import pytest
import torch

import jsd_inputs
from parity_util import TOL, rel_fro

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 << 20  # the array size the header states


def _existing(problem_kw, inputs, chunk_rows):
    from lm_head_jsd_gb300 import FusedLinearJSD

    x_s, w_s, x_t, w_t, labels = inputs
    run = FusedLinearJSD(x_s.shape[0], x_s.shape[1], x_t.shape[1], w_s.shape[0], x_s.dtype,
                         chunk_rows=chunk_rows, device=x_s.device, **problem_kw)
    out = run.forward(x_s, w_s, x_t, w_t, labels)
    torch.cuda.synchronize()
    return out


def _noalloc(problem_kw, inputs):
    from lm_head_jsd_gb300 import _lib

    x_s, w_s, x_t, w_t, labels = inputs
    bt, h_s = x_s.shape
    v = w_s.shape[0]
    dt = "bf16" if x_s.dtype == torch.bfloat16 else "fp32"
    p = _lib.make_problem(bt, h_s, x_t.shape[1], v, dt, **problem_kw)
    n_loss = bt if problem_kw.get("reduction") == "none" else 1
    loss = torch.empty(n_loss, dtype=torch.float32, device=x_s.device)
    gi = torch.empty(bt, h_s, dtype=x_s.dtype, device=x_s.device)
    gw = torch.empty(v, h_s, dtype=x_s.dtype, device=x_s.device)
    _lib.fljsd_forward_noalloc(p, x_s, w_s, x_t, w_t, labels, None, loss, gi, gw)
    torch.cuda.synchronize()
    # the chunking it chose: the planner limited to the array
    plan = _lib.fljsd_plan(p, 2 * SCRATCH_BYTES)
    assert plan.workspace_bytes <= SCRATCH_BYTES
    return (loss, gi, gw), int(plan.chunk_rows)


def _check(got, ref, dtype, what):
    tol_loss, tol_grad = TOL[dtype]
    e = rel_fro(got[0].double().cpu().numpy(), ref[0].double().cpu().numpy())
    assert e <= tol_loss, f"{what}: loss {e:.3g}"
    for name, g, r in (("grad_input", got[1], ref[1]), ("grad_weight", got[2], ref[2])):
        e = rel_fro(g.double().cpu().numpy(), r.double().cpu().numpy())
        assert e <= tol_grad, f"{what}: {name} {e:.3g}"


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    dev = "cuda:0"
    # call 1: the whole batch fits in one chunk of the fixed array
    w1 = jsd_inputs.custom("noalloc1", 41, 300, 64, 5000, "bf16", ignore_frac=0.1)
    in1 = jsd_inputs.make_inputs(w1, dev)
    kw1 = dict(beta=0.5, temperature=1.0, reduction="batchmean")
    got1, c1 = _noalloc(kw1, in1)
    assert c1 == 300
    _check(got1, _existing(kw1, in1, c1), "bf16", "call 1")

    # call 2: another problem, large enough that the array forces several chunks
    w2 = jsd_inputs.custom("noalloc2", 42, 1024, 128, 40000, "bf16", ignore_frac=0.05,
                           beta=0.1, temperature=2.0)
    in2 = jsd_inputs.make_inputs(w2, dev)
    kw2 = dict(beta=0.1, temperature=2.0, reduction="none")
    got2, c2 = _noalloc(kw2, in2)
    assert c2 < 1024
    _check(got2, _existing(kw2, in2, c2), "bf16", "call 2")


def test_noalloc_rejects_problems_beyond_the_array():
    from lm_head_jsd_gb300 import _lib

    fake = 1 << 20  # aligned; never dereferenced because the call is rejected first
    p = _lib.make_problem(16, 64, 64, 20_000_000, "bf16")  # one row needs 80 MB
    st = _lib.fljsd_forward_noalloc(p, fake, fake, fake, fake, None, None, fake, fake, fake,
                                    check=False)
    assert st == 3  # FLJSD_ERR_WORKSPACE
