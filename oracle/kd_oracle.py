"""fp64 CPU oracle for the top-K KL distillation loss.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
benchmark's CPU-baseline leg may import this module; the product path never
calls it, and it shares no code with the CUDA path.

What it computes is the plain dense definition of the loss that the fused
chunked kernels must reproduce.  The write-ups of "Efficient Knowledge
Distillation for LLMs: Offline Top-K Logits and a Fused Chunked KL Loss" state
the method in words only:
  * the teacher's top 100 predictions per position are cached once and the
    student trains against that cache alone (ai2day.live story, "What did the
    researchers change?"; elseif.net summary, second paragraph);
  * the KL divergence between teacher and student is computed chunk by chunk
    over the sequence, each chunk calculated and discarded, with the backward
    pass recomputing what it needs (same ai2day.live section);
  * the chunked loss is mathematically equivalent to the dense one (iwenai.com
    essay, paragraph after "Enter a new approach") and must be validated
    against the dense baseline (elseif.net summary, last paragraph);
  * rare-token probabilities outside the top K are discarded (elseif.net
    summary, third paragraph), so the teacher distribution is renormalised
    over the K cached entries.
So the oracle is the dense computation itself, in float64, blocked over token
rows only (rows are independent): no vocabulary tiling, no fusion, no
recomputation.

Definitions (natural log, temperature T shared by teacher and student):
  p_r      = softmax over the K cached entries of (teacher logit / T)
  z        = h W^T,  s = z / T,  lse_r = logsumexp over the vocabulary of s_r
  loss_r   = sum_k p_rk (log p_rk - (s_{r,idx_rk} - lse_r))
  loss     = sum over valid rows of loss_r / N_valid            (0 if N_valid = 0)
  dL/dz_rv = (softmax(s_r)_v - sum_{k: idx_rk = v} p_rk) / (T N_valid)
  grad_h   = (dL/dz) W,   grad_W = (dL/dz)^T h
Readings where the pages are silent (each also listed with the design notes):
  * no T^2 factor; mean over valid tokens;
  * a duplicate index adds its probabilities (scatter-add);
  * an index outside [0, V) is dropped from the teacher distribution (as if its
    logit were -inf) and raises FLAG_INDEX_RANGE;
  * a -inf teacher logit gives p = 0 and a zero term;
  * a valid row whose in-range teacher logits include NaN or +inf, or hold no
    finite value, is excluded like a masked row (no loss, zero gradient, not
    counted in N_valid) and raises FLAG_BAD_TEACHER;
  * mask 1 = valid; masked rows' data is never used.
"""
from __future__ import annotations

import numpy as np

FLAG_INDEX_RANGE = 1
FLAG_BAD_TEACHER = 2


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def teacher_distribution(topk_idx, topk_logit, mask, V, T):
    """Teacher probabilities renormalised over the cached entries.

    Returns (p [N,K] float64, valid [N] bool, flags int).  p is 0 for dropped
    entries and for rows that are not valid."""
    idx = np.asarray(topk_idx, dtype=np.int64)
    lg = _f64(topk_logit)
    N, K = idx.shape
    valid = np.ones(N, dtype=bool) if mask is None else (np.asarray(mask) != 0)
    in_range = (idx >= 0) & (idx < V)
    flags = 0
    if np.any(valid[:, None] & ~in_range):
        flags |= FLAG_INDEX_RANGE
    with np.errstate(invalid="ignore"):
        nan_or_pinf = in_range & (np.isnan(lg) | (lg == np.inf))
        finite = in_range & np.isfinite(lg)
    bad = valid & (nan_or_pinf.any(axis=1) | ~finite.any(axis=1))
    if bad.any():
        flags |= FLAG_BAD_TEACHER
    valid = valid & ~bad
    p = np.zeros((N, K), dtype=np.float64)
    rows = np.nonzero(valid)[0]
    if rows.size:
        x = np.where(in_range[rows], lg[rows] / T, -np.inf)
        m = x.max(axis=1, keepdims=True)
        e = np.exp(x - m)
        p[rows] = e / e.sum(axis=1, keepdims=True)
    return p, valid, flags


def _plogp(p):
    out = np.zeros_like(p)
    pos = p > 0
    out[pos] = p[pos] * np.log(p[pos])
    return out.sum(axis=1)


def _row_block(H, W, idx, p, valid, T, n_valid):
    """Dense forward and dL/dz for one block of rows.  Returns (lse, loss_rows, G).

    Rows that are not valid are replaced by zeros first, so nothing they hold
    (NaN included) reaches a result."""
    H = np.where(valid[:, None], H, 0.0)
    S = (H @ W.T) / T
    m = S.max(axis=1, keepdims=True)
    lse = (m + np.log(np.exp(S - m).sum(axis=1, keepdims=True)))[:, 0]
    V = W.shape[0]
    in_range = (idx >= 0) & (idx < V)
    safe = np.where(in_range, idx, 0)
    s_idx = np.take_along_axis(S, safe, axis=1)
    pk = np.where(in_range, p, 0.0)
    loss_rows = _plogp(pk) - (pk * (s_idx - lse[:, None])).sum(axis=1)
    loss_rows = np.where(valid, loss_rows, 0.0)
    G = np.exp(S - lse[:, None])
    r = np.repeat(np.arange(H.shape[0]), idx.shape[1])
    np.add.at(G, (r, safe.reshape(-1)), -pk.reshape(-1))
    G /= (T * max(n_valid, 1))
    G[~valid] = 0.0
    return lse, loss_rows, G


def fwd_bwd(h, W, topk_idx, topk_logit, mask, T, block_rows=256, want_grads=True, n_norm=None):
    """Dense loss, grad_h and grad_W in float64.

    h [N,d], W [V,d] are the exact values the kernels see (bf16 or fp32
    widened to float64).  Returns a dict with loss, grad_h, grad_W, lse,
    loss_rows, valid, n_valid, flags.  Rows are processed in blocks of
    block_rows; the result does not depend on that size beyond rounding.

    n_norm: the divisor of the mean, N_valid of these rows by default.  When
    a batch is split into token shards, the batch's loss is still the mean
    over all of its valid tokens, so each shard divides by the batch's
    N_valid: the shards' losses and grad_W then add up to the batch's."""
    H = _f64(h)
    Wd = _f64(W)
    N, d = H.shape
    V = Wd.shape[0]
    p, valid, flags = teacher_distribution(topk_idx, topk_logit, mask, V, T)
    n_valid = int(valid.sum())
    div = n_valid if n_norm is None else int(n_norm)
    lse = np.full(N, np.nan)
    loss_rows = np.zeros(N)
    grad_h = np.zeros((N, d)) if want_grads else None
    grad_W = np.zeros((V, d)) if want_grads else None
    idx = np.asarray(topk_idx, dtype=np.int64)
    for r0 in range(0, N, block_rows):
        r1 = min(N, r0 + block_rows)
        v = valid[r0:r1]
        if not v.any():
            continue
        l_b, lr_b, G = _row_block(H[r0:r1], Wd, idx[r0:r1], p[r0:r1], v, T, div)
        lse[r0:r1] = np.where(v, l_b, np.nan)
        loss_rows[r0:r1] = lr_b
        if want_grads:
            grad_h[r0:r1] = G @ Wd
            grad_W += G.T @ np.where(v[:, None], H[r0:r1], 0.0)
    loss = float(loss_rows.sum() / div) if div > 0 else 0.0
    return dict(loss=loss, grad_h=grad_h, grad_W=grad_W, lse=lse, loss_rows=loss_rows,
                valid=valid, n_valid=n_valid, flags=flags, p=p)


def fwd(h, W, topk_idx, topk_logit, mask, T, block_rows=256, n_norm=None):
    """Loss only (same definition as fwd_bwd)."""
    return fwd_bwd(h, W, topk_idx, topk_logit, mask, T, block_rows, want_grads=False,
                   n_norm=n_norm)


def teacher_plogp(p):
    """Per-row sum_k p_k ln p_k of teacher probabilities p [N,K] (0 ln 0 = 0):
    the teacher-entropy term of loss_r."""
    return _plogp(_f64(p))


def grad_logits(h, W, topk_idx, topk_logit, mask, T, block_rows=256):
    """The dense gradient of the loss with respect to the student logits,
    dL/dz [N,V] in float64 (zero rows for rows that are not valid), computed
    block by block exactly as inside fwd_bwd.  grad_h = (dL/dz) W and
    grad_W = (dL/dz)^T h.  Returns a dict with G, lse, p, valid, n_valid."""
    H = _f64(h)
    Wd = _f64(W)
    N = H.shape[0]
    V = Wd.shape[0]
    p, valid, _ = teacher_distribution(topk_idx, topk_logit, mask, V, T)
    n_valid = int(valid.sum())
    idx = np.asarray(topk_idx, dtype=np.int64)
    G = np.zeros((N, V))
    lse = np.full(N, np.nan)
    for r0 in range(0, N, block_rows):
        r1 = min(N, r0 + block_rows)
        v = valid[r0:r1]
        if not v.any():
            continue
        l_b, _, G_b = _row_block(H[r0:r1], Wd, idx[r0:r1], p[r0:r1], v, T, n_valid)
        lse[r0:r1] = np.where(v, l_b, np.nan)
        G[r0:r1] = G_b
    return dict(G=G, lse=lse, p=p, valid=valid, n_valid=n_valid)


def sampled_rows(h, W, topk_idx, topk_logit, mask, T, rows, block_rows=64):
    """Per-row results for a subset of rows, each computed on its own.

    Every row's loss term, lse and grad_h row depend only on that row (and on
    N_valid, which needs the teacher data of all rows but no student logits),
    so the full-size problems can be checked row by row.  Returns a dict with
    rows, valid, lse, loss_rows, grad_h (rows of the full grad_h), n_valid."""
    Wd = _f64(W)
    V = Wd.shape[0]
    p_all, valid_all, flags = teacher_distribution(topk_idx, topk_logit, mask, V, T)
    n_valid = int(valid_all.sum())
    rows = np.asarray(rows, dtype=np.int64)
    idx = np.asarray(topk_idx, dtype=np.int64)
    lse = np.full(rows.size, np.nan)
    loss_rows = np.zeros(rows.size)
    grad_h = np.zeros((rows.size, Wd.shape[1]))
    for b0 in range(0, rows.size, block_rows):
        rr = rows[b0:b0 + block_rows]
        v = valid_all[rr]
        l_b, lr_b, G = _row_block(_f64(h[rr]), Wd, idx[rr], p_all[rr], v, T, n_valid)
        lse[b0:b0 + rr.size] = np.where(v, l_b, np.nan)
        loss_rows[b0:b0 + rr.size] = lr_b
        grad_h[b0:b0 + rr.size] = G @ Wd
    return dict(rows=rows, valid=valid_all[rows], lse=lse, loss_rows=loss_rows,
                grad_h=grad_h, n_valid=n_valid, flags=flags)


def grad_W_rows(h, W, topk_idx, topk_logit, mask, T, vocab_rows, lse):
    """Rows v of grad_W = (dL/dz)^T h, each computed on its own.

    Column v of dL/dz needs z_rv = h_r . W_v for every token r and the
    per-token lse (from fwd), so one grad_W row costs O(N d) once lse is
    known.  lse is the oracle's own (NaN for rows that are not valid)."""
    H = _f64(h)
    Wd = _f64(W)
    V = Wd.shape[0]
    p, valid, _ = teacher_distribution(topk_idx, topk_logit, mask, V, T)
    n_valid = int(valid.sum())
    idx = np.asarray(topk_idx, dtype=np.int64)
    in_range = (idx >= 0) & (idx < V)
    Hv = np.where(valid[:, None], H, 0.0)
    lse_v = np.where(valid, lse, 0.0)
    vocab_rows = np.asarray(vocab_rows, dtype=np.int64)
    S = (Hv @ Wd[vocab_rows].T) / T                       # [N, n]
    G = np.exp(S - lse_v[:, None])
    for j, v in enumerate(vocab_rows):
        hit = in_range & (idx == v)
        G[:, j] -= (p * hit).sum(axis=1)
    G /= (T * max(n_valid, 1))
    G[~valid] = 0.0
    return G.T @ Hv
