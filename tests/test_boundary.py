"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point its header declares, plans chunks as documented, and rejects
bad arguments synchronously with a status before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fljsd.h")


@pytest.fixture(scope="module")
def L():
    from conftest import build_library

    build_library()
    from lm_head_jsd_gb300 import _lib

    return _lib


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fljsd_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("fljsd_plan", "fljsd_forward", "fljsd_backward", "fljsd_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    lib = ctypes.CDLL(L.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r"\bT (fljsd_\w+)", out))
    assert set(_declared_functions()) <= exported


def test_status_strings(L):
    assert L.fljsd_status_string(0) == "ok"
    assert L.fljsd_status_string(3) == "workspace too small"
    assert L.fljsd_status_string(99) == "unknown status"


def test_plan_single_chunk_and_memory_accounting(L):
    # PR 1352 "Details", memory table: the two logits tensors take 2*C*V*s bytes
    # and loss_1d takes BT*4 bytes.
    p = L.make_problem(8192, 4096, 4096, 128256, "bf16")
    plan = L.fljsd_plan(p, 0)
    assert plan.chunk_rows == 8192 and plan.num_chunks == 1 and plan.ld == 128256
    assert plan.logits_bytes == 2 * 8192 * 128256 * 2
    assert plan.workspace_bytes >= plan.logits_bytes + 8192 * 4
    # beyond the logits: loss_1d (BT*4), the pass-1 partials of both models
    # (8 bytes per row per 128 columns each) and alignment
    partials = 2 * 8192 * (-(-128256 // 128)) * 8
    assert plan.stats_bytes >= partials + 8192 * 4
    extra = plan.workspace_bytes - plan.logits_bytes
    assert partials + 8192 * 4 <= extra < partials + 8192 * 4 + 4096
    # ld is padded to a multiple of 8 elements (16-byte rows in bf16)
    plan = L.fljsd_plan(L.make_problem(64, 128, 128, 1000, "fp32"), 0)
    assert plan.ld == 1000
    plan = L.fljsd_plan(L.make_problem(64, 128, 128, 1001, "bf16"), 0)
    assert plan.ld == 1008 and plan.logits_bytes == 2 * 64 * 1008 * 2


def test_planner_fits_free_memory(L):
    p = L.make_problem(8192, 4096, 4096, 128256, "bf16")
    one_chunk = L.fljsd_plan(p, 0).workspace_bytes
    plan = L.fljsd_plan(p, one_chunk)  # only half of it may be used
    assert plan.chunk_rows % 128 == 0 and 0 < plan.chunk_rows < 8192
    assert plan.workspace_bytes <= one_chunk // 2
    assert plan.num_chunks == -(-8192 // plan.chunk_rows)
    bigger = L.fljsd_plan(p, 4 * one_chunk)
    assert bigger.chunk_rows == 8192
    # explicit chunk rows are honoured and clamped to bt
    p.chunk_rows = 512
    assert L.fljsd_plan(p, 0).chunk_rows == 512
    p.chunk_rows = 100000
    assert L.fljsd_plan(p, 0).chunk_rows == 8192
    # not even one row fits
    p.chunk_rows = 0
    with pytest.raises(L.FljsdError) as e:
        L.fljsd_plan(p, 1024)
    assert e.value.status == 3


def test_planner_fp32_accumulator_only_charged_to_chunked_plans(L):
    """With FLJSD_FLAG_ACCUM_FP32 the V x H fp32 grad_weight accumulator is
    needed only when there is more than one chunk (PR 1429's accum_dtype
    option accumulates across chunks). A budget that holds the one-chunk
    workspace but not the accumulator must give one chunk, not an error."""
    p = L.make_problem(64, 4096, 4096, 128256, "bf16", accum_fp32=True)
    single = L.fljsd_plan(p, 0)
    assert single.chunk_rows == 64 and single.num_chunks == 1
    acc_bytes = 128256 * 4096 * 4
    assert single.workspace_bytes < acc_bytes  # the one-chunk plan carries no accumulator
    plan = L.fljsd_plan(p, 2 * single.workspace_bytes)  # half of it is the budget
    assert plan.chunk_rows == 64 and plan.num_chunks == 1
    assert plan.workspace_bytes == single.workspace_bytes
    # the same budget without the flag gives the same plan
    q = L.make_problem(64, 4096, 4096, 128256, "bf16")
    assert L.fljsd_plan(q, 2 * single.workspace_bytes).workspace_bytes == single.workspace_bytes
    # a multi-chunk plan does carry it: it needs more than the accumulator
    big = L.make_problem(8192, 4096, 4096, 128256, "bf16", accum_fp32=True)
    one_chunk = L.fljsd_plan(big, 0).workspace_bytes
    chunked = L.fljsd_plan(big, one_chunk)  # half of one chunk's workspace
    assert chunked.num_chunks > 1 and chunked.workspace_bytes > acc_bytes
    assert chunked.workspace_bytes <= one_chunk // 2
    # a budget below the accumulator cannot hold any chunked plan
    with pytest.raises(L.FljsdError) as e:
        L.fljsd_plan(big, acc_bytes)
    assert e.value.status == 3


@pytest.mark.parametrize("field,value", [
    ("bt", 0), ("h_s", -1), ("h_t", 0), ("v", 0), ("dtype", 7), ("reduction", 9),
    ("beta", 1.5), ("beta", -0.1), ("beta", float("nan")), ("temperature", 0.0),
    ("temperature", -1.0), ("temperature", float("inf")), ("temperature", float("nan")),
    ("chunk_rows", -4),
])
def test_plan_rejects_bad_problems(L, field, value):
    p = L.make_problem(16, 32, 32, 100, "bf16")
    setattr(p, field, value)
    with pytest.raises(L.FljsdError) as e:
        L.fljsd_plan(p, 0)
    assert e.value.status == 1


@pytest.mark.parametrize("field,value", [("bt", (1 << 30) + 1), ("v", (1 << 30) + 1),
                                         ("h_s", (1 << 20) + 1), ("h_t", (1 << 20) + 1)])
def test_plan_reports_sizes_beyond_the_kernels(L, field, value):
    """Valid problems beyond the kernels' index ranges (32-bit vector indices
    along a row, grid limits) are refused with FLJSD_ERR_UNSUPPORTED, not
    launched; the largest supported sizes plan."""
    p = L.make_problem(16, 32, 32, 100, "bf16")
    setattr(p, field, value)
    with pytest.raises(L.FljsdError) as e:
        L.fljsd_plan(p, 0)
    assert e.value.status == 2
    setattr(p, field, value - 1)
    assert L.fljsd_plan(p, 0).chunk_rows > 0


@pytest.mark.parametrize("bt,h,v", [((1 << 30) + 1, 32, 100), (16, (1 << 20) + 1, 100),
                                    (16, 32, (1 << 30) + 1)])
def test_ce_plan_reports_sizes_beyond_the_kernels(L, bt, h, v):
    with pytest.raises(L.FljsdError) as e:
        L.fljsd_ce_plan(L.make_ce_problem(bt, h, v, "bf16"), 0)
    assert e.value.status == 2


C_CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "fljsd.h"

int main(void) {
  fljsd_problem p;
  memset(&p, 0, sizeof p);
  p.bt = 8192; p.h_s = 4096; p.h_t = 4096; p.v = 128256;
  p.dtype = FLJSD_BF16; p.reduction = FLJSD_RED_BATCHMEAN;
  p.beta = 0.5f; p.temperature = 1.0f; p.ignore_index = -100;
  fljsd_plan_t plan;
  fljsd_status st = fljsd_plan(&p, 0, &plan);
  printf("%d %lld %lld %zu\n", (int)st, (long long)plan.chunk_rows,
         (long long)plan.num_chunks, plan.workspace_bytes);
  p.beta = 2.0f;
  st = fljsd_plan(&p, 0, &plan);
  printf("%d %s\n", (int)st, fljsd_status_string(st));
  return 0;
}
"""


def test_plain_c_client_links_and_plans(L, tmp_path):
    """The boundary is plain C: a C99 program that includes only fljsd.h
    compiles (-Wall -Werror), links against libfljsd.so and plans the headline
    problem (one chunk, the workspace the Python binding reports) and gets a
    synchronous INVALID_ARG for beta outside [0, 1]. No device call is made."""
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(L.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I",
                    os.path.join(ROOT, "include"), str(src), "-o", str(exe), "-L", libdir,
                    "-lfljsd", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    st, chunk, nchunks, ws = out[0].split()
    ref = L.fljsd_plan(L.make_problem(8192, 4096, 4096, 128256, "bf16"), 0)
    assert (int(st), int(chunk), int(nchunks), int(ws)) == (0, 8192, 1, ref.workspace_bytes)
    assert out[1].split()[0] == "1"


def _fake(addr=1 << 20):
    return addr  # an aligned, never dereferenced address


def test_forward_argument_checks_need_no_device(L):
    p = L.make_problem(16, 32, 32, 100, "bf16")
    plan = L.fljsd_plan(p, 0)
    good = dict(x_s=_fake(), w_s=_fake(), x_t=_fake(), w_t=_fake(), labels=None, row_grad=None,
                loss=_fake(), grad_input=_fake(), grad_weight=_fake(), workspace=_fake())

    def call(ws_bytes=plan.workspace_bytes, problem=p, pl=plan, **over):
        a = dict(good, **over)
        return L.fljsd_forward(problem, pl, a["x_s"], a["w_s"], a["x_t"], a["w_t"], a["labels"],
                               a["row_grad"], a["loss"], a["grad_input"], a["grad_weight"],
                               a["workspace"], workspace_bytes=ws_bytes, stream=0, check=False)

    for k in ("x_s", "w_s", "x_t", "w_t", "loss", "grad_input", "grad_weight", "workspace"):
        assert call(**{k: None}) == 1, k
        assert call(**{k: _fake() + 8}) == 1, k  # misaligned
    assert call(labels=_fake() + 4) == 1
    assert call(ws_bytes=plan.workspace_bytes - 1) == 3
    other = L.fljsd_plan(L.make_problem(16, 32, 32, 200, "bf16"), 0)
    assert call(pl=other) == 1  # plan made for another problem
    bad = L.make_problem(16, 32, 32, 100, "bf16", beta=2.0)
    assert call(problem=bad) == 1


@pytest.mark.parametrize("fn", ["jsd_logspace", "tvd"])
def test_distance_argument_checks_need_no_device(L, fn):
    """fljsd_jsd_logspace / fljsd_tvd refuse bad calls on the host, before any
    launch: sizes (INVALID_ARG for <= 0, UNSUPPORTED above 2^31), dtype,
    reduction, null or unaligned pointers, beta, and a short workspace."""
    ws = L.fljsd_rows_workspace_bytes(16)

    def call(rows=16, v=100, dtype="bf16", reduction="sum", x=_fake(), y=_fake(), loss=_fake(),
             grad=_fake(), workspace=_fake(), ws_bytes=ws, beta=0.5, labels=None):
        if fn == "jsd_logspace":
            return L.fljsd_jsd_logspace(rows, v, dtype, beta, reduction, -100, x, y, labels, loss,
                                        grad, workspace, workspace_bytes=ws_bytes, stream=0,
                                        check=False)
        return L.fljsd_tvd(rows, v, dtype, reduction, -100, x, y, labels, loss, grad, workspace,
                           workspace_bytes=ws_bytes, stream=0, check=False)

    assert call(rows=0) == 1 and call(v=0) == 1 and call(rows=-3) == 1
    assert call(rows=(1 << 31) + 1) == 2 and call(v=(1 << 31) + 1) == 2
    assert call(x=0) == 1 and call(y=0) == 1 and call(loss=0) == 1 and call(grad=0) == 1
    assert call(workspace=0) == 1
    assert call(x=_fake() + 8) == 1 and call(grad=_fake() + 4) == 1 and call(loss=_fake() + 2) == 1
    assert call(labels=_fake() + 8) == 1
    assert call(ws_bytes=ws - 1) == 3
    if fn == "jsd_logspace":
        assert call(beta=1.5) == 1 and call(beta=float("nan")) == 1


def test_backward_argument_checks_need_no_device(L):
    p = L.make_problem(16, 32, 32, 100, "bf16")
    assert L.fljsd_backward(p, None, _fake(), _fake(), stream=0, check=False) == 1
    assert L.fljsd_backward(p, _fake(), None, _fake(), stream=0, check=False) == 1
    assert L.fljsd_backward(p, _fake(), _fake() + 2, _fake(), stream=0, check=False) == 1


def test_package_has_no_cpu_fallback():
    """The product package never imports the oracle, and nothing in it computes
    the loss with torch: every step runs in libfljsd.so."""
    pkg = os.path.join(ROOT, "lm_head_jsd_gb300")
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            src = open(os.path.join(pkg, fn)).read()
            assert "oracle" not in src, fn
            for forbidden in ("log_softmax", "torch.matmul", "softmax(", " @ "):
                assert forbidden not in src, (fn, forbidden)
