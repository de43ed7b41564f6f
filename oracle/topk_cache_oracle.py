"""fp64 CPU oracle for building the offline teacher top-K cache.

TEST INFRASTRUCTURE ONLY.  Only the tests and the benchmark's CPU-baseline leg
may import this module; the product path never calls it, and it shares no
code with the CUDA path.

The write-ups of "Efficient Knowledge Distillation for LLMs: Offline Top-K
Logits and a Fused Chunked KL Loss" describe the offline stage in words: the
teacher runs once over the corpus and its top 100 predictions per position
are written to the cache, after which the teacher is switched off (ai2day.live
story, "What did the researchers change?"; aiphreaks.com summary, bullet on
the top-100 cache; elseif.net summary, second paragraph).  So the cache entry
of position r holds the K largest teacher logits z_r = h_r W^T with their
vocabulary indices.

What the pages leave open, and the reading taken here:
  * the cached values are the raw logits z (the loss renormalises them over
    the K entries with its own temperature, so a shift or a log-softmax would
    give the same teacher distribution);
  * ties: among equal logits the lower vocabulary index ranks first, so the
    selection and its order are unique;
  * the K entries are stored in rank order: logit descending, index ascending
    among equal logits;
  * a NaN logit ranks below every number (it is never preferred to a real
    logit) and, among NaNs, the lower index first.

The oracle is that definition written out: z in float64, blocked over rows
only, then each row ordered by the key (logit descending, index ascending).
"""
from __future__ import annotations

import numpy as np


def rank_order(z_row):
    """Vocabulary indices of one row of logits in rank order: logit
    descending, lower index first among equal logits, NaN last."""
    z = np.asarray(z_row, dtype=np.float64)
    v = np.arange(z.shape[0])
    nan = np.isnan(z)
    # np.lexsort sorts by the last key first: NaN flag, then -z, then index
    return np.lexsort((v, -np.where(nan, 0.0, z), nan))


def topk_cache(h, W, K, block_rows=256):
    """The top-K cache of teacher hidden states h [N, d] against the teacher's
    LM head W [V, d]: (topk_idx [N, K] int32, topk_logit [N, K] float64)."""
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    N = h.shape[0]
    V = W.shape[0]
    if not 1 <= K <= V:
        raise ValueError("need 1 <= K <= V")
    idx = np.zeros((N, K), dtype=np.int32)
    val = np.zeros((N, K), dtype=np.float64)
    for r0 in range(0, N, block_rows):
        Z = h[r0:r0 + block_rows] @ W.T
        for j in range(Z.shape[0]):
            order = rank_order(Z[j])[:K]
            idx[r0 + j] = order
            val[r0 + j] = Z[j, order]
    return idx, val


def row_logits(h, W, rows):
    """Full logit rows z[rows, :] in float64."""
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    return h[np.asarray(rows)] @ W.T
