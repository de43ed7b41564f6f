"""fp64 CPU oracles (test infrastructure only; the product path never imports
them): the top-K KL distillation loss, and the offline teacher top-K cache it
reads."""
from .kd_oracle import (FLAG_BAD_TEACHER, FLAG_INDEX_RANGE, fwd, fwd_bwd, grad_W_rows,
                        sampled_rows, teacher_distribution)
from .topk_cache_oracle import logits_at, rank_order, row_logits, topk_cache

__all__ = ["FLAG_BAD_TEACHER", "FLAG_INDEX_RANGE", "fwd", "fwd_bwd", "grad_W_rows",
           "sampled_rows", "teacher_distribution", "topk_cache", "rank_order", "logits_at",
           "row_logits"]
