"""fp64 CPU oracle for the full-vocabulary (K = V) distillation loss.

TEST INFRASTRUCTURE ONLY.  Only the tests and the benchmark's CPU-baseline leg
may import this module; the product path never calls it, and it shares no
code with the CUDA path.

The write-ups of "Efficient Knowledge Distillation for LLMs: Offline Top-K
Logits and a Fused Chunked KL Loss" contrast the offline top-K cache with
online distillation, where the teacher stays resident and its full output
distribution is used every step (ai2day.live story, the comparison table's
"online distillation" row; elseif.net summary, third paragraph: the cache
drops the rare-token probabilities that the full distribution keeps).  This
is that loss on the full vocabulary: the teacher's logits come from its final
hidden states and LM head in the same pass, nothing is truncated.

Definitions (natural log, temperature T shared by teacher and student):
  t = h_t W_t^T / T,   s = h_s W_s^T / T
  p_r = softmax(t_r),  log q_r = s_r - logsumexp(s_r)
  loss = (1 / N_valid) * sum over valid rows of sum_v p_rv (log p_rv - log q_rv)
  dL/dz_s = (softmax(s_r) - p_r) / (T N_valid),  grad_h = (dL/dz_s) W_s,
  grad_W = (dL/dz_s)^T h_s   (the teacher is not trained)
Readings where the pages are silent, as for the top-K loss: no T^2 factor,
mean over valid tokens (mask 1 = valid, NULL = all), N_valid = 0 gives zero
loss and gradients, outputs are overwritten.  Teacher and student share the
vocabulary; their hidden sizes may differ.

The oracle is that definition in float64, blocked over rows only.
"""
from __future__ import annotations

import numpy as np


def _log_softmax(x):
    m = x.max(axis=1, keepdims=True)
    return x - (m + np.log(np.exp(x - m).sum(axis=1, keepdims=True)))


def full_kl_fwd_bwd(h_s, W_s, h_t, W_t, mask, T, block_rows=256, want_grads=True):
    """Returns dict(loss, grad_h [N, d_s], grad_W [V, d_s], loss_rows [N],
    lse_s [N] (logsumexp of s), lse_t [N] (logsumexp of t), valid [N] bool,
    n_valid)."""
    h_s = np.asarray(h_s, dtype=np.float64)
    W_s = np.asarray(W_s, dtype=np.float64)
    h_t = np.asarray(h_t, dtype=np.float64)
    W_t = np.asarray(W_t, dtype=np.float64)
    N = h_s.shape[0]
    V = W_s.shape[0]
    valid = np.ones(N, dtype=bool) if mask is None else np.asarray(mask) != 0
    n_valid = int(valid.sum())
    loss_rows = np.zeros(N)
    lse_s = np.zeros(N)
    lse_t = np.zeros(N)
    grad_h = np.zeros_like(h_s) if want_grads else None
    grad_W = np.zeros_like(W_s) if want_grads else None
    for r0 in range(0, N, block_rows):
        rows = np.arange(r0, min(N, r0 + block_rows))
        rows = rows[valid[rows]]
        if rows.size == 0:
            continue
        t = (h_t[rows] @ W_t.T) / T
        s = (h_s[rows] @ W_s.T) / T
        logp = _log_softmax(t)
        logq = _log_softmax(s)
        p = np.exp(logp)
        loss_rows[rows] = (p * (logp - logq)).sum(axis=1)
        smax = s.max(axis=1)
        lse_s[rows] = smax + np.log(np.exp(s - smax[:, None]).sum(axis=1))
        tmax = t.max(axis=1)
        lse_t[rows] = tmax + np.log(np.exp(t - tmax[:, None]).sum(axis=1))
        if want_grads:
            G = (np.exp(logq) - p) / (T * n_valid)
            grad_h[rows] = G @ W_s
            grad_W += G.T @ h_s[rows]
    loss = float(loss_rows[valid].sum() / n_valid) if n_valid > 0 else 0.0
    return dict(loss=loss, grad_h=grad_h, grad_W=grad_W, loss_rows=loss_rows, lse_s=lse_s,
                lse_t=lse_t, valid=valid, n_valid=n_valid)


def full_kl_grad_logits(h_s, W_s, h_t, W_t, mask, T):
    """The dense gradient of the full-vocabulary loss with respect to the
    student logits z_s = h_s W_s^T: dL/dz_s = (softmax(s) - softmax(t)) /
    (T N_valid), zero rows for masked rows.  Returns dict(G [N, V], q (student
    softmax), p (teacher softmax), valid, n_valid); q and p are zero on masked
    rows."""
    h_s = np.asarray(h_s, dtype=np.float64)
    W_s = np.asarray(W_s, dtype=np.float64)
    h_t = np.asarray(h_t, dtype=np.float64)
    W_t = np.asarray(W_t, dtype=np.float64)
    N, V = h_s.shape[0], W_s.shape[0]
    valid = np.ones(N, dtype=bool) if mask is None else np.asarray(mask) != 0
    n_valid = int(valid.sum())
    q = np.zeros((N, V))
    p = np.zeros((N, V))
    rows = np.nonzero(valid)[0]
    if rows.size:
        q[rows] = np.exp(_log_softmax((h_s[rows] @ W_s.T) / T))
        p[rows] = np.exp(_log_softmax((h_t[rows] @ W_t.T) / T))
    G = (q - p) / (T * max(n_valid, 1))
    return dict(G=G, q=q, p=p, valid=valid, n_valid=n_valid)


def full_kl_sampled_rows(h_s, W_s, h_t, W_t, mask, T, rows, block_rows=64):
    """Per-row results of the full loss for the given rows only: loss_rows,
    lse_s and grad_h rows, with N_valid over the whole batch.  Masked rows
    give a zero loss term and a zero grad_h row, as in full_kl_fwd_bwd.  The
    rows are taken block_rows at a time."""
    valid = (np.ones(np.asarray(h_s).shape[0], dtype=bool) if mask is None
             else np.asarray(mask) != 0)
    n_valid = int(valid.sum())
    rows = np.asarray(rows)
    Ws = np.asarray(W_s, dtype=np.float64)
    Wt = np.asarray(W_t, dtype=np.float64)
    loss_rows = np.zeros(rows.size)
    lse_s = np.zeros(rows.size)
    grad_h = np.zeros((rows.size, Ws.shape[1]))
    for b0 in range(0, rows.size, block_rows):
        rr = rows[b0:b0 + block_rows]
        hs = np.asarray(h_s, dtype=np.float64)[rr]
        ht = np.asarray(h_t, dtype=np.float64)[rr]
        t = (ht @ Wt.T) / T
        s = (hs @ Ws.T) / T
        logp = _log_softmax(t)
        logq = _log_softmax(s)
        p = np.exp(logp)
        loss_rows[b0:b0 + rr.size] = (p * (logp - logq)).sum(axis=1)
        smax = s.max(axis=1)
        lse_s[b0:b0 + rr.size] = smax + np.log(np.exp(s - smax[:, None]).sum(axis=1))
        G = (np.exp(logq) - p) / (T * max(n_valid, 1))
        grad_h[b0:b0 + rr.size] = G @ Ws
    v = valid[rows]
    grad_h[~v] = 0.0
    loss_rows[~v] = 0.0
    return dict(loss_rows=loss_rows, lse_s=lse_s, grad_h=grad_h, valid=v, n_valid=n_valid)


def full_kl_grad_W_rows(h_s, W_s, h_t, W_t, mask, T, vocab_rows, lse_s, lse_t,
                        block_rows=4096):
    """Rows vocab_rows of grad_W = (dL/dz_s)^T h_s, given every row's lse_s and
    lse_t (from full_kl_fwd_bwd): column v of dL/dz_s is
    (exp(s_v - lse_s) - exp(t_v - lse_t)) / (T N_valid) over the valid rows,
    so only those columns of both products are formed."""
    h_s = np.asarray(h_s, dtype=np.float64)
    h_t = np.asarray(h_t, dtype=np.float64)
    vr = np.asarray(vocab_rows)
    Ws = np.asarray(W_s, dtype=np.float64)[vr]
    Wt = np.asarray(W_t, dtype=np.float64)[vr]
    N = h_s.shape[0]
    valid = np.ones(N, dtype=bool) if mask is None else np.asarray(mask) != 0
    n_valid = int(valid.sum())
    out = np.zeros((vr.size, h_s.shape[1]))
    if n_valid == 0:
        return out
    for r0 in range(0, N, block_rows):
        rows = np.arange(r0, min(N, r0 + block_rows))
        rows = rows[valid[rows]]
        if rows.size == 0:
            continue
        s = (h_s[rows] @ Ws.T) / T
        t = (h_t[rows] @ Wt.T) / T
        G = (np.exp(s - lse_s[rows, None]) - np.exp(t - lse_t[rows, None])) / (T * n_valid)
        out += G.T @ h_s[rows]
    return out
