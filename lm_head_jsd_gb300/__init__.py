"""GB300 (sm_103a) fused-linear Jensen-Shannon distillation loss.

The compute path is libfljsd.so (CUDA kernels behind the C ABI declared in
include/fljsd.h). This package is its binding: ``_lib`` mirrors the C entry
points by name, ``api`` adds torch allocation and an autograd Function.
"""
from ._lib import (  # noqa: F401
    FljsdError,
    fljsd_backward,
    fljsd_ce_forward,
    fljsd_ce_plan,
    make_ce_problem,
    fljsd_forward,
    fljsd_forward_noalloc,
    fljsd_gemm_bf16,
    fljsd_jsd_logspace,
    fljsd_rows_workspace_bytes,
    fljsd_scale,
    fljsd_tvd,
    fljsd_launch_count,
    fljsd_launch_count_reset,
    fljsd_plan,
    fljsd_status_string,
    fljsd_trace_enable,
    fljsd_trace_read,
    fljsd_trace_reset,
    fljsd_workspace_status,
    make_problem,
)
from .api import (  # noqa: F401
    FusedLinearCrossEntropy,
    FusedLinearJSD,
    fused_linear_cross_entropy,
    fused_linear_jsd,
    jsd_logspace,
    tvd,
)

LIB_PATH = _lib.LIB_PATH
