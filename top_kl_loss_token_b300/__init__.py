"""Fused chunked top-K KL distillation loss for B300 (sm_103a)."""
