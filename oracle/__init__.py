"""fp64 CPU oracle for the fused top-K forward-KL loss (test infrastructure only)."""
from .fkl_oracle import (  # noqa: F401
    teacher_distribution, row_valid, student_lse, forward, backward,
    rows_forward_backward, dW_rows, kl_rows_from_logits, teacher_topk,
    forward_mix, backward_mix,
)
