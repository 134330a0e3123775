"""CPU float64 oracle of the fused-linear JSD loss (test infrastructure only).

Only tests, the smoke check and the CPU-baseline leg of the benchmark use this
package. The product library never imports it, and it imports nothing from
the product library.
"""
from .fljsd_oracle import (  # noqa: F401
    REDUCTIONS,
    bf16_round,
    dist_zero_masks,
    fljsd_from_logits,
    fljsd_ref,
    fljsd_rows_ref,
    flce_ref,
    jsd_logspace_ref,
    jsd_rows,
    log_softmax_rows,
    logits,
    row_weights,
    tie_mask,
    tvd_ref,
    zero_masks,
)
