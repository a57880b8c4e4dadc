"""CPU FP64 oracle for chunked linear cross-entropy (test infrastructure only).

Only tests, the smoke check and the benchmark's CPU-baseline leg may import
this package.  The GPU library shares no code with it and never calls it.
"""
from .lce_oracle import (IGNORE_INDEX, as_f64, backward, check_labels, count_valid, forward,  # noqa: F401
                         fused, grad_W_columns, grad_scale_per_row, logits, logsumexp_rows, rows_forward,
                         rows_grad_X, softmax_minus_onehot, target_logits, valid_mask)
