"""The tensor-core GEMM building block (fljsd_gemm_bf16) against a plain PyTorch
fp32 reference of the same contraction, for every operand layout the path uses,
ragged shapes, multi-tile shapes and the accumulate (beta = 1) epilogue."""
import pytest
import torch

pytestmark = pytest.mark.gpu

SHAPES = [
    # (m, n, k)
    (1, 8, 8), (7, 9, 24), (128, 256, 64), (300, 1000, 200), (129, 257, 65),
    (1024, 2048, 1024), (64, 4096, 2048), (2000, 512, 4096),
]


def _operand(mn_major, outer, inner, gen):
    """bf16 matrix stored [outer x inner] row-major with values in N(0, 1), as a
    view of storage whose row stride is a multiple of 8 elements; the padding
    holds NaN so that reading it would show."""
    ld = -(-inner // 8) * 8
    buf = torch.full((outer, ld), float("nan"), dtype=torch.bfloat16, device="cuda")
    buf[:, :inner] = torch.randn(outer, inner, generator=gen, device="cuda").to(torch.bfloat16)
    return buf[:, :inner], ld


def _ref(a, a_mn, b, b_mn):
    A = a.float().t() if a_mn else a.float()  # [m x k]
    B = b.float().t() if b_mn else b.float()  # [n x k]
    return A @ B.t()


@pytest.mark.parametrize("flags", [0, 1], ids=["pairs", "single"])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1), (1, 0)])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_gemm_layouts(a_mn, b_mn, shape, flags, monkeypatch):
    from lm_head_jsd_gb300 import fljsd_gemm_bf16

    if flags == 0:  # CTA pairs at every contraction depth
        monkeypatch.setenv("FLJSD_GEMM_PAIR", "2")

    m, n, k = shape
    g = torch.Generator(device="cuda").manual_seed(m * 7 + n * 3 + k)
    a, lda = _operand(a_mn, k if a_mn else m, m if a_mn else k, g)
    b, ldb = _operand(b_mn, k if b_mn else n, n if b_mn else k, g)
    ldd = -(-n // 8) * 8
    dbuf = torch.empty(m, ldd, dtype=torch.bfloat16, device="cuda")
    d = dbuf[:, :n]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fljsd_gemm_bf16(a, lda, a_mn, b, ldb, b_mn, d, ldd, m, n, k, 0, status, flags)
    torch.cuda.synchronize()
    assert status.item() == 0
    ref = _ref(a, a_mn, b, b_mn)
    err = (d.float() - ref).norm() / ref.norm()
    assert err < 4e-3, float(err)
    # accumulate: D = D + A.B^T
    d0 = d.clone()
    fljsd_gemm_bf16(a, lda, a_mn, b, ldb, b_mn, d, ldd, m, n, k, 1, status, flags)
    torch.cuda.synchronize()
    ref2 = d0.float() + ref
    err = (d.float() - ref2).norm() / ref2.norm()
    assert err < 4e-3, float(err)


def test_gemm_strided_output_and_guard():
    """Output with a row stride larger than n: the padding columns and the rows
    past m are never written."""
    from lm_head_jsd_gb300 import fljsd_gemm_bf16

    m, n, k, ldd = 200, 1000, 320, 1032
    g = torch.Generator(device="cuda").manual_seed(5)
    a = torch.randn(m, k, generator=g, device="cuda").to(torch.bfloat16)
    b = torch.randn(n, k, generator=g, device="cuda").to(torch.bfloat16)
    buf = torch.full((m + 3, ldd), 7.0, dtype=torch.bfloat16, device="cuda")
    fljsd_gemm_bf16(a, k, 0, b, k, 0, buf, ldd, m, n, k, 0)
    torch.cuda.synchronize()
    assert torch.all(buf[:, n:] == 7.0) and torch.all(buf[m:] == 7.0)
    ref = a.float() @ b.float().t()
    err = (buf[:m, :n].float() - ref).norm() / ref.norm()
    assert err < 4e-3


def test_gemm_rejects_bad_arguments():
    from lm_head_jsd_gb300 import fljsd_gemm_bf16

    a = torch.zeros(16, 16, dtype=torch.bfloat16, device="cuda")
    assert fljsd_gemm_bf16(a, 16, 0, a, 16, 0, a, 16, 16, 16, 0, check=False) == 1  # k = 0
    assert fljsd_gemm_bf16(a, 12, 0, a, 16, 0, a, 16, 16, 16, 12, check=False) == 1  # lda % 8
    assert fljsd_gemm_bf16(a, 16, 2, a, 16, 0, a, 16, 16, 16, 16, check=False) == 1
    assert fljsd_gemm_bf16(a, 16, 0, a, 16, 0, a, 16, 16, 16, 16, flags=4, check=False) == 1


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1), (1, 0)])
@pytest.mark.parametrize("shape", [(1000, 777, 300), (256, 512, 64), (384, 1000, 1000),
                                   (4096, 4096, 512)],
                         ids=lambda s: "x".join(map(str, s)))
def test_gemm_pairs_and_single_ctas_agree_bitwise(a_mn, b_mn, shape, monkeypatch):
    """A CTA pair computes a 256-row tile with one MMA instruction over both
    CTAs' shared memory; one CTA computes 128 rows. The products and their
    fp32 accumulation order are the same, so both schedules give identical
    bits (including an odd m-block count, whose last pair has an empty half)."""
    from lm_head_jsd_gb300 import fljsd_gemm_bf16

    monkeypatch.setenv("FLJSD_GEMM_PAIR", "2")  # pairs at every contraction depth

    m, n, k = shape
    g = torch.Generator(device="cuda").manual_seed(11 + m + n + k)
    a, lda = _operand(a_mn, k if a_mn else m, m if a_mn else k, g)
    b, ldb = _operand(b_mn, k if b_mn else n, n if b_mn else k, g)
    ldd = -(-n // 8) * 8
    d0 = torch.empty(m, ldd, dtype=torch.bfloat16, device="cuda")
    d1 = torch.empty(m, ldd, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fljsd_gemm_bf16(a, lda, a_mn, b, ldb, b_mn, d0, ldd, m, n, k, 0, status, 0)
    fljsd_gemm_bf16(a, lda, a_mn, b, ldb, b_mn, d1, ldd, m, n, k, 0, status, 1)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(d0[:, :n], d1[:, :n])
    ref = _ref(a, a_mn, b, b_mn)
    assert ((d0[:, :n].float() - ref).norm() / ref.norm()).item() < 4e-3


@pytest.mark.parametrize("flags", [0, 1], ids=["pairs", "single"])
@pytest.mark.parametrize("a_mn,b_mn", [(1, 1), (0, 0), (0, 1)])
@pytest.mark.parametrize("shape", [(1000, 777, 128), (300, 1000, 640), (129, 4096, 2048),
                                   (5000, 4096, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_gemm_accumulate_prefetch_matches_plain_loads(a_mn, b_mn, shape, flags, monkeypatch):
    if flags == 0:  # CTA pairs at every contraction depth
        monkeypatch.setenv("FLJSD_GEMM_PAIR", "2")
    """The accumulating epilogue reads the old values from slabs copied ahead by
    TMA (shallow, middle and deep operand rings by contraction length); with the
    copy turned off it reads them with plain loads. Same arithmetic, so the
    results agree bitwise; padding columns and rows past m stay untouched."""
    from lm_head_jsd_gb300 import fljsd_gemm_bf16

    m, n, k = shape
    g = torch.Generator(device="cuda").manual_seed(m + n + k)
    a, lda = _operand(a_mn, k if a_mn else m, m if a_mn else k, g)
    b, ldb = _operand(b_mn, k if b_mn else n, n if b_mn else k, g)
    ldd = -(-n // 8) * 8 + 8
    base = torch.full((m + 2, ldd), 3.0, dtype=torch.bfloat16, device="cuda")
    base[:m, :n] = torch.randn(m, n, generator=g, device="cuda").to(torch.bfloat16)
    outs = []
    for pf in ("1", "0"):
        monkeypatch.setenv("FLJSD_GEMM_PREFETCH", pf)
        buf = base.clone()
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        fljsd_gemm_bf16(a, lda, a_mn, b, ldb, b_mn, buf, ldd, m, n, k, 1, status, flags)
        torch.cuda.synchronize()
        assert status.item() == 0
        assert torch.all(buf[:, n:] == 3.0) and torch.all(buf[m:] == 3.0)
        outs.append(buf)
    assert torch.equal(outs[0], outs[1])
    ref = base[:m, :n].float() + _ref(a, a_mn, b, b_mn)
    err = (outs[0][:m, :n].float() - ref).norm() / ref.norm()
    assert err < 4e-3, float(err)


@pytest.mark.parametrize("flags", [0, 1], ids=["pairs", "single"])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("shape", [(1000, 1000, 128), (129, 4096, 640), (300, 264, 4096)],
                         ids=lambda s: "x".join(map(str, s)))
def test_gemm_staged_output_matches_plain_stores(a_mn, b_mn, shape, flags, monkeypatch):
    if flags == 0:  # CTA pairs at every contraction depth
        monkeypatch.setenv("FLJSD_GEMM_PAIR", "2")
    """A plain (non-accumulating) bf16 output goes through shared-memory staging
    buffers and TMA stores; with staging turned off each thread stores its row.
    Same rounding, so the results agree bitwise; the stores are clipped at the
    output's bounds (padding columns and rows past m untouched)."""
    from lm_head_jsd_gb300 import fljsd_gemm_bf16

    m, n, k = shape
    g = torch.Generator(device="cuda").manual_seed(m * 3 + n + k)
    a, lda = _operand(a_mn, k if a_mn else m, m if a_mn else k, g)
    b, ldb = _operand(b_mn, k if b_mn else n, n if b_mn else k, g)
    ldd = n + 16
    outs = []
    for so in ("1", "0"):
        monkeypatch.setenv("FLJSD_GEMM_STAGE_OUT", so)
        buf = torch.full((m + 2, ldd), 5.0, dtype=torch.bfloat16, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        fljsd_gemm_bf16(a, lda, a_mn, b, ldb, b_mn, buf, ldd, m, n, k, 0, status, flags)
        torch.cuda.synchronize()
        assert status.item() == 0
        assert torch.all(buf[:, n:] == 5.0) and torch.all(buf[m:] == 5.0)
        outs.append(buf)
    assert torch.equal(outs[0], outs[1])
    ref = _ref(a, a_mn, b, b_mn)
    err = (outs[0][:m, :n].float() - ref).norm() / ref.norm()
    assert err < 4e-3, float(err)
