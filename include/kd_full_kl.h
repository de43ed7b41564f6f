/*
 * kd_full_kl.h -- the full-vocabulary (K = V) distillation loss on B300
 * (sm_103a): the teacher's logits are computed from its final hidden states
 * and LM head in the same pass, so nothing of its distribution is truncated.
 *
 * "Efficient Knowledge Distillation for LLMs: Offline Top-K Logits and a
 * Fused Chunked KL Loss" contrasts its offline top-K cache with online
 * distillation, where the teacher stays resident and its whole output
 * distribution is used at every step (ai2day.live story, the comparison
 * table's "online distillation" row; elseif.net summary, third paragraph: the
 * cache drops the rare-token probabilities).  This call computes that loss
 * with the same fused, chunked machinery as kd_topk_kl_fwd_bwd (kd_topk_kl.h):
 * no N x V grid is ever materialised.
 *
 * Definitions (natural log; T shared by teacher and student):
 *   t = h_t W_t^T / T,  s = h_s W_s^T / T,  p = softmax(t),  q = softmax(s)
 *   loss     = (1 / N_valid) sum over valid rows of sum_v p_v (log p_v - log q_v)
 *   dL/dz_s  = (q - p) / (T N_valid);  grad_h = (dL/dz_s) W_s,  grad_W = (dL/dz_s)^T h_s
 * The teacher is frozen (no teacher gradients).  There is no T^2 factor;
 * N_valid = 0 gives loss 0 and zero gradients.
 *
 * Layouts (row-major, contiguous, 16-byte aligned device buffers, bf16):
 *   h_s [N, d_s], W_s [V, d_s]   student final hidden states and LM head
 *   h_t [N, d_t], W_t [V, d_t]   teacher final hidden states and LM head
 *   mask [N] uint8 (1 = valid; NULL = every row valid); masked rows' data is
 *   never read for a result
 *   loss [1] fp32, grad_h [N, d_s] fp32, grad_W [V, d_s] fp32: overwritten
 * d_s and d_t must be multiples of 8 (tensor-memory-accelerator rows).
 *
 * Ownership and execution as in kd_topk_kl.h: the caller owns every buffer
 * including the workspace; nothing is allocated; the call is stream-ordered
 * and asynchronous; the status covers host-side checks and launch errors;
 * device-side problems are ORed into *dev_err_flags (KD_FLAG_TIMEOUT).
 */
#ifndef KD_FULL_KL_H
#define KD_FULL_KL_H

#include "kd_topk_kl.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Workspace bytes for these sizes (chunk <= 0: the default chunk); 0 for
 * invalid sizes.  Per chunk: both models' exponential tiles (2 x chunk x V
 * bf16), five per-(row, 128-column block) statistics, the gathered hidden
 * states; per row: the valid-row map, lse and loss terms.
 */
size_t kd_full_kl_workspace_bytes(int64_t N, int64_t d_s, int64_t d_t, int64_t V, int64_t chunk);

/*
 * The chunk used when a call passes chunk <= 0: equal chunks of a multiple of
 * 128 rows, small enough that both models' exponential tiles stay near 8 GiB
 * and that both models' hidden states of a chunk (chunk x (d_s + d_t) bf16)
 * stay within 48 MiB, the part of L2 that holds data re-read by every tile.
 */
int64_t kd_full_kl_default_chunk(int64_t N, int64_t d_s, int64_t d_t, int64_t V);

/*
 * Loss, grad_h and grad_W of the full-vocabulary loss.  Per chunk of valid
 * rows: one tensor-core pass computes each tile's teacher and student logits
 * (both into tensor memory) and keeps per-block statistics and the stored
 * exponentials of both; a row kernel combines them into the exact KL and the
 * gradient tile (q - p) / (T N_valid); two persistent tensor-core GEMMs give
 * grad_h and grad_W.
 * Errors: KD_ERR_INVALID_ARG (NULL pointer, N < 0, d_s, d_t or V < 1, T not
 * finite or <= 0, misaligned buffer), KD_ERR_UNSUPPORTED (d_s or d_t not a
 * multiple of 8, sizes beyond 2^31), KD_ERR_WORKSPACE, KD_ERR_CUDA.
 */
kd_status kd_full_kl_fwd_bwd(const void* h_s, const void* W_s, const void* h_t, const void* W_t,
                             const uint8_t* mask, int64_t N, int64_t d_s, int64_t d_t, int64_t V,
                             float T, int64_t chunk, float* loss, float* grad_h, float* grad_W,
                             void* workspace, size_t ws_bytes, uint32_t* dev_err_flags,
                             cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KD_FULL_KL_H */
