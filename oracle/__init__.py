"""fp64 CPU oracles (test infrastructure only; the product path never imports
them): the top-K KL distillation loss, the offline teacher top-K cache it
reads, and the full-vocabulary (K = V) loss with the teacher computed in the
same pass."""
from .kd_oracle import (FLAG_BAD_TEACHER, FLAG_INDEX_RANGE, fwd, fwd_bwd, grad_logits,
                        grad_W_rows, sampled_rows, teacher_distribution, teacher_plogp)
from .topk_cache_oracle import rank_order, row_logits, topk_cache
from .full_kl_oracle import (full_kl_fwd_bwd, full_kl_grad_W_rows, full_kl_grad_logits,
                             full_kl_sampled_rows)

__all__ = ["FLAG_BAD_TEACHER", "FLAG_INDEX_RANGE", "fwd", "fwd_bwd", "grad_logits",
           "grad_W_rows", "sampled_rows", "teacher_distribution", "teacher_plogp", "topk_cache",
           "rank_order", "row_logits", "full_kl_fwd_bwd", "full_kl_grad_logits",
           "full_kl_sampled_rows"]
