"""Failure detection without a GPU fault: every mbarrier wait of the GEMM is
bounded. With FLJSD_GEMM_TEST_STALL the copy warp issues nothing, so the first
wait of the MMA warp expires after 50 ms; the kernel must report
FLJSD_ERR_TIMEOUT in the device status word, free its tensor memory and exit,
and the context must stay usable for the next call."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("acc", [0, 1], ids=["store", "accumulate"])
@pytest.mark.parametrize("pairs", [True, False], ids=["pairs", "single"])
def test_gemm_wait_timeout_is_reported_and_the_context_survives(pairs, acc, monkeypatch):
    """With acc = 1 the stored output is read ahead by the prefetch warp, whose
    ring of slabs fills and whose waits then expire as well. In a CTA pair
    both CTAs' waits expire (each on its own clock) and both leave through
    the cluster barrier at the exit."""
    from lm_head_jsd_gb300 import _lib

    if pairs:  # CTA pairs at this contraction depth too
        monkeypatch.setenv("FLJSD_GEMM_PAIR", "2")
    m, n, k = 512, 512, 256
    g = torch.Generator(device="cuda").manual_seed(3)
    a = torch.randn(m, k, generator=g, device="cuda").to(torch.bfloat16)
    b = torch.randn(n, k, generator=g, device="cuda").to(torch.bfloat16)
    d0 = torch.randn(m, n, generator=g, device="cuda").to(torch.bfloat16)
    d = d0.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flags = _lib.FLJSD_GEMM_TEST_STALL | (0 if pairs else _lib.FLJSD_GEMM_SINGLE_CTA)
    _lib.fljsd_gemm_bf16(a, k, 0, b, k, 0, d, n, m, n, k, acc, status, flags)
    torch.cuda.synchronize()
    assert status.item() == 5  # FLJSD_ERR_TIMEOUT
    # the same GEMM, unstalled, on the same context
    d.copy_(d0)
    status.zero_()
    _lib.fljsd_gemm_bf16(a, k, 0, b, k, 0, d, n, m, n, k, acc, status,
                         0 if pairs else _lib.FLJSD_GEMM_SINGLE_CTA)
    torch.cuda.synchronize()
    assert status.item() == 0
    ref = a.float() @ b.float().t() + (d0.float() if acc else 0.0)
    assert ((d.float() - ref).norm() / ref.norm()).item() < 4e-3


def test_forward_reports_ok_in_the_workspace_status():
    import jsd_inputs
    from lm_head_jsd_gb300 import FusedLinearJSD, fljsd_workspace_status

    w = jsd_inputs.custom("status", 61, 256, 64, 3000, "bf16")
    x_s, w_s, x_t, w_t = (t.cuda() for t in jsd_inputs.make_inputs(w, "cpu")[:4])
    run = FusedLinearJSD(256, 64, 64, 3000, torch.bfloat16)
    run.forward(x_s, w_s, x_t, w_t)
    assert fljsd_workspace_status(run.plan, run.workspace) == 0
