"""fp64 CPU oracle for the top-K KL distillation loss (test infrastructure only;
the product path never imports it)."""
from .kd_oracle import (FLAG_BAD_TEACHER, FLAG_INDEX_RANGE, fwd, fwd_bwd, grad_W_rows,
                        sampled_rows, teacher_distribution)

__all__ = ["FLAG_BAD_TEACHER", "FLAG_INDEX_RANGE", "fwd", "fwd_bwd", "grad_W_rows",
           "sampled_rows", "teacher_distribution"]
