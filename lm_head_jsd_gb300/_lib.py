"""ctypes binding of libfljsd.so (argument marshalling only).

The functions carry the names of the C entry points in include/fljsd.h. Tensor
arguments are torch tensors whose device pointers are passed through; no
arithmetic of the loss happens in Python. If the shared library is missing the
import fails: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfljsd.so")

FLJSD_OK = 0
STATUS_NAMES = {0: "FLJSD_OK", 1: "FLJSD_ERR_INVALID_ARG", 2: "FLJSD_ERR_UNSUPPORTED",
                3: "FLJSD_ERR_WORKSPACE", 4: "FLJSD_ERR_CUDA", 5: "FLJSD_ERR_TIMEOUT"}
DTYPES = {"fp32": 0, "bf16": 1}
REDUCTIONS = {"none": 0, "sum": 1, "mean": 2, "batchmean": 3}
KERNEL_KINDS = {"gemm_logits": 0, "jsd_rows": 1, "gemm_grad_input": 2,
                "gemm_grad_weight": 3, "small": 4}


class FljsdError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} "
                         f"({fljsd_status_string(status)})")


class fljsd_problem(ctypes.Structure):
    _fields_ = [("bt", ctypes.c_int64), ("h_s", ctypes.c_int64), ("h_t", ctypes.c_int64),
                ("v", ctypes.c_int64), ("dtype", ctypes.c_int32), ("reduction", ctypes.c_int32),
                ("beta", ctypes.c_float), ("temperature", ctypes.c_float),
                ("ignore_index", ctypes.c_int64), ("chunk_rows", ctypes.c_int64),
                ("flags", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class fljsd_ce_problem(ctypes.Structure):
    _fields_ = [("bt", ctypes.c_int64), ("h", ctypes.c_int64), ("v", ctypes.c_int64),
                ("dtype", ctypes.c_int32), ("reduction", ctypes.c_int32),
                ("ignore_index", ctypes.c_int64), ("chunk_rows", ctypes.c_int64),
                ("label_smoothing", ctypes.c_float), ("lse_square_scale", ctypes.c_float),
                ("softcap", ctypes.c_float), ("flags", ctypes.c_int32)]


FLJSD_FLAG_T2 = 1
FLJSD_FLAG_ACCUM_FP32 = 2


class fljsd_plan_t(ctypes.Structure):
    _fields_ = [("chunk_rows", ctypes.c_int64), ("num_chunks", ctypes.c_int64),
                ("ld", ctypes.c_int64), ("workspace_bytes", ctypes.c_size_t),
                ("logits_bytes", ctypes.c_size_t), ("stats_bytes", ctypes.c_size_t),
                ("status_offset", ctypes.c_size_t)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python lm_head_jsd_gb300/build.py` (there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    lib.fljsd_plan.argtypes = [ctypes.POINTER(fljsd_problem), ctypes.c_size_t,
                               ctypes.POINTER(fljsd_plan_t)]
    lib.fljsd_plan.restype = ctypes.c_int
    lib.fljsd_forward.argtypes = [ctypes.POINTER(fljsd_problem), ctypes.POINTER(fljsd_plan_t),
                                  P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
    lib.fljsd_forward.restype = ctypes.c_int
    lib.fljsd_forward_noalloc.argtypes = [ctypes.POINTER(fljsd_problem), P, P, P, P, P, P, P, P,
                                          P, P]
    lib.fljsd_forward_noalloc.restype = ctypes.c_int
    lib.fljsd_backward.argtypes = [ctypes.POINTER(fljsd_problem), P, P, P, P]
    lib.fljsd_backward.restype = ctypes.c_int
    lib.fljsd_workspace_status.argtypes = [ctypes.POINTER(fljsd_plan_t), P, P,
                                           ctypes.POINTER(ctypes.c_int32)]
    lib.fljsd_workspace_status.restype = ctypes.c_int
    lib.fljsd_gemm_bf16.argtypes = [P, ctypes.c_int64, ctypes.c_int32, P, ctypes.c_int64,
                                    ctypes.c_int32, P, ctypes.c_int64, ctypes.c_int64,
                                    ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, P,
                                    ctypes.c_int32, P]
    lib.fljsd_gemm_bf16.restype = ctypes.c_int
    lib.fljsd_rows_workspace_bytes.argtypes = [ctypes.c_int64]
    lib.fljsd_rows_workspace_bytes.restype = ctypes.c_size_t
    lib.fljsd_jsd_logspace.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                       ctypes.c_float, ctypes.c_int32, ctypes.c_int64, P, P, P,
                                       P, P, P, ctypes.c_size_t, P]
    lib.fljsd_jsd_logspace.restype = ctypes.c_int
    lib.fljsd_tvd.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                              ctypes.c_int64, P, P, P, P, P, P, ctypes.c_size_t, P]
    lib.fljsd_tvd.restype = ctypes.c_int
    lib.fljsd_scale.argtypes = [ctypes.c_int32, P, ctypes.c_int64, P, P]
    lib.fljsd_scale.restype = ctypes.c_int
    lib.fljsd_ce_plan.argtypes = [ctypes.POINTER(fljsd_ce_problem), ctypes.c_size_t,
                                  ctypes.POINTER(fljsd_plan_t)]
    lib.fljsd_ce_plan.restype = ctypes.c_int
    lib.fljsd_ce_forward.argtypes = [ctypes.POINTER(fljsd_ce_problem),
                                     ctypes.POINTER(fljsd_plan_t), P, P, P, P, P, P, P,
                                     ctypes.c_size_t, P]
    lib.fljsd_ce_forward.restype = ctypes.c_int
    lib.fljsd_status_string.argtypes = [ctypes.c_int]
    lib.fljsd_status_string.restype = ctypes.c_char_p
    lib.fljsd_launch_count.argtypes = []
    lib.fljsd_launch_count.restype = ctypes.c_int64
    lib.fljsd_launch_count_reset.argtypes = []
    lib.fljsd_launch_count_reset.restype = None
    lib.fljsd_trace_enable.argtypes = [ctypes.c_int32]
    lib.fljsd_trace_enable.restype = ctypes.c_int
    lib.fljsd_trace_reset.argtypes = []
    lib.fljsd_trace_reset.restype = ctypes.c_int
    lib.fljsd_trace_read.argtypes = [ctypes.c_int32, ctypes.POINTER(ctypes.c_double),
                                     ctypes.POINTER(ctypes.c_int64)]
    lib.fljsd_trace_read.restype = ctypes.c_int
    return lib


lib = _load()


def _ptr(t) -> int | None:
    """Device (or host) address of a tensor, None for None; ints pass through."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_problem(bt, h_s, h_t, v, dtype="bf16", reduction="batchmean", beta=0.5,
                 temperature=1.0, ignore_index=-100, chunk_rows=0, t2_scale=False,
                 accum_fp32=False) -> fljsd_problem:
    flags = (FLJSD_FLAG_T2 if t2_scale else 0) | (FLJSD_FLAG_ACCUM_FP32 if accum_fp32 else 0)
    return fljsd_problem(bt, h_s, h_t, v, DTYPES[dtype] if isinstance(dtype, str) else dtype,
                         REDUCTIONS[reduction] if isinstance(reduction, str) else reduction,
                         beta, temperature, ignore_index, chunk_rows, flags, 0)


def fljsd_status_string(status: int) -> str:
    return lib.fljsd_status_string(status).decode()


def fljsd_plan(problem: fljsd_problem, free_hbm_bytes: int = 0) -> fljsd_plan_t:
    plan = fljsd_plan_t()
    st = lib.fljsd_plan(ctypes.byref(problem), free_hbm_bytes, ctypes.byref(plan))
    if st != FLJSD_OK:
        raise FljsdError(st, "fljsd_plan")
    return plan


def fljsd_forward(problem, plan, x_s, w_s, x_t, w_t, labels, row_grad, loss, grad_input,
                  grad_weight, workspace, workspace_bytes=None, stream=None, check=True) -> int:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    st = lib.fljsd_forward(ctypes.byref(problem), ctypes.byref(plan), _ptr(x_s), _ptr(w_s),
                           _ptr(x_t), _ptr(w_t), _ptr(labels), _ptr(row_grad), _ptr(loss),
                           _ptr(grad_input), _ptr(grad_weight), _ptr(workspace),
                           workspace_bytes, _stream(stream))
    if check and st != FLJSD_OK:
        raise FljsdError(st, "fljsd_forward")
    return st


def fljsd_forward_noalloc(problem, x_s, w_s, x_t, w_t, labels, row_grad, loss, grad_input,
                          grad_weight, stream=None, check=True) -> int:
    """fljsd_forward with the library's fixed device scratch instead of a
    caller-provided workspace (for callers that cannot allocate)."""
    st = lib.fljsd_forward_noalloc(ctypes.byref(problem), _ptr(x_s), _ptr(w_s), _ptr(x_t),
                                   _ptr(w_t), _ptr(labels), _ptr(row_grad), _ptr(loss),
                                   _ptr(grad_input), _ptr(grad_weight), _stream(stream))
    if check and st != FLJSD_OK:
        raise FljsdError(st, "fljsd_forward_noalloc")
    return st


def fljsd_backward(problem, grad_output, grad_input, grad_weight, stream=None,
                   check=True) -> int:
    st = lib.fljsd_backward(ctypes.byref(problem), _ptr(grad_output), _ptr(grad_input),
                            _ptr(grad_weight), _stream(stream))
    if check and st != FLJSD_OK:
        raise FljsdError(st, "fljsd_backward")
    return st


def fljsd_workspace_status(plan, workspace, stream=None) -> int:
    out = ctypes.c_int32()
    st = lib.fljsd_workspace_status(ctypes.byref(plan), _ptr(workspace), _stream(stream),
                                    ctypes.byref(out))
    if st != FLJSD_OK:
        raise FljsdError(st, "fljsd_workspace_status")
    return out.value


FLJSD_GEMM_SINGLE_CTA = 1
FLJSD_GEMM_TEST_STALL = 2


def fljsd_gemm_bf16(a, lda, a_mn, b, ldb, b_mn, d, ldd, m, n, k, accumulate=0, status=None,
                    flags=0, stream=None, check=True) -> int:
    st = lib.fljsd_gemm_bf16(_ptr(a), lda, a_mn, _ptr(b), ldb, b_mn, _ptr(d), ldd, m, n, k,
                             accumulate, _ptr(status), flags, _stream(stream))
    if check and st != FLJSD_OK:
        raise FljsdError(st, "fljsd_gemm_bf16")
    return st


def _dt(dtype):
    return DTYPES[dtype] if isinstance(dtype, str) else int(dtype)


def _red(reduction):
    return REDUCTIONS[reduction] if isinstance(reduction, str) else int(reduction)


def fljsd_rows_workspace_bytes(rows: int) -> int:
    return lib.fljsd_rows_workspace_bytes(rows)


def fljsd_jsd_logspace(rows, v, dtype, beta, reduction, ignore_index, input, target, labels,
                       loss, grad_input, workspace, workspace_bytes=None, stream=None,
                       check=True) -> int:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    st = lib.fljsd_jsd_logspace(rows, v, _dt(dtype), beta, _red(reduction), ignore_index,
                                _ptr(input), _ptr(target), _ptr(labels), _ptr(loss),
                                _ptr(grad_input), _ptr(workspace), workspace_bytes,
                                _stream(stream))
    if check and st != FLJSD_OK:
        raise FljsdError(st, "fljsd_jsd_logspace")
    return st


def fljsd_tvd(rows, v, dtype, reduction, ignore_index, p, q, labels, loss, grad_p, workspace,
              workspace_bytes=None, stream=None, check=True) -> int:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    st = lib.fljsd_tvd(rows, v, _dt(dtype), _red(reduction), ignore_index, _ptr(p), _ptr(q),
                       _ptr(labels), _ptr(loss), _ptr(grad_p), _ptr(workspace), workspace_bytes,
                       _stream(stream))
    if check and st != FLJSD_OK:
        raise FljsdError(st, "fljsd_tvd")
    return st


def fljsd_scale(dtype, x, n, grad_output, stream=None, check=True) -> int:
    st = lib.fljsd_scale(_dt(dtype), _ptr(x), n, _ptr(grad_output), _stream(stream))
    if check and st != FLJSD_OK:
        raise FljsdError(st, "fljsd_scale")
    return st


def make_ce_problem(bt, h, v, dtype="bf16", reduction="mean", ignore_index=-100, chunk_rows=0,
                    label_smoothing=0.0, lse_square_scale=0.0, softcap=0.0,
                    accum_fp32=False) -> fljsd_ce_problem:
    return fljsd_ce_problem(bt, h, v, _dt(dtype), _red(reduction), ignore_index, chunk_rows,
                            label_smoothing, lse_square_scale, softcap,
                            FLJSD_FLAG_ACCUM_FP32 if accum_fp32 else 0)


def fljsd_ce_plan(problem, free_hbm_bytes: int = 0) -> fljsd_plan_t:
    plan = fljsd_plan_t()
    st = lib.fljsd_ce_plan(ctypes.byref(problem), free_hbm_bytes, ctypes.byref(plan))
    if st != FLJSD_OK:
        raise FljsdError(st, "fljsd_ce_plan")
    return plan


def fljsd_ce_forward(problem, plan, x, w, labels, loss, grad_input, grad_weight, workspace,
                     workspace_bytes=None, stream=None, check=True) -> int:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    st = lib.fljsd_ce_forward(ctypes.byref(problem), ctypes.byref(plan), _ptr(x), _ptr(w),
                              _ptr(labels), _ptr(loss), _ptr(grad_input), _ptr(grad_weight),
                              _ptr(workspace), workspace_bytes, _stream(stream))
    if check and st != FLJSD_OK:
        raise FljsdError(st, "fljsd_ce_forward")
    return st


def fljsd_launch_count() -> int:
    return lib.fljsd_launch_count()


def fljsd_launch_count_reset() -> None:
    lib.fljsd_launch_count_reset()


def fljsd_trace_enable(max_launches: int) -> None:
    st = lib.fljsd_trace_enable(max_launches)
    if st != FLJSD_OK:
        raise FljsdError(st, "fljsd_trace_enable")


def fljsd_trace_reset() -> None:
    lib.fljsd_trace_reset()


def fljsd_trace_read(kind) -> tuple[float, int]:
    k = KERNEL_KINDS[kind] if isinstance(kind, str) else kind
    ms = ctypes.c_double()
    n = ctypes.c_int64()
    st = lib.fljsd_trace_read(k, ctypes.byref(ms), ctypes.byref(n))
    if st != FLJSD_OK:
        raise FljsdError(st, "fljsd_trace_read")
    return ms.value, n.value
