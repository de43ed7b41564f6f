/*
 * kd_topk_cache.h -- building the offline teacher top-K cache on B300 (sm_103a).
 *
 * The distillation method of "Efficient Knowledge Distillation for LLMs:
 * Offline Top-K Logits and a Fused Chunked KL Loss" runs the teacher once over
 * the corpus and keeps only its top 100 predictions per position, after which
 * the teacher is switched off (ai2day.live story, "What did the researchers
 * change?"; aiphreaks.com summary, bullet on the top-100 cache; elseif.net
 * summary, second paragraph).  This call produces that cache from the
 * teacher's final hidden states and LM head: for every position r, the K
 * largest logits z_r = h_r W^T and their vocabulary indices -- the
 * (topk_idx, topk_logit) input of kd_topk_kl_fwd_bwd.
 *
 * Ranking: logit descending; among equal logits the lower vocabulary index
 * first; a NaN logit ranks below every number (among NaNs, the lower index
 * first) and raises KD_FLAG_BAD_TEACHER.  -0.0 and +0.0 are equal.  The K
 * entries of a row are written in rank order.  The logits are those of the
 * tensor-core product (bf16 inputs, fp32 accumulation), written as fp32.
 *
 * Layouts (row-major, contiguous, 16-byte aligned device buffers):
 *   h          [N, d]  bf16   teacher final hidden states
 *   W          [V, d]  bf16   teacher LM-head weight (nn.Linear layout)
 *   topk_idx   [N, K]  int32  written
 *   topk_logit [N, K]  fp32   written
 * d must be a multiple of 8; 1 <= K <= min(V, KD_MAX_K).
 *
 * Ownership and execution: as for kd_topk_kl_fwd_bwd (kd_topk_kl.h): the
 * caller owns every buffer including the workspace, the library allocates
 * nothing, the call is stream-ordered and asynchronous, and the returned
 * status covers only host-side checks and launch errors.
 */
#ifndef KD_TOPK_CACHE_H
#define KD_TOPK_CACHE_H

#include "kd_topk_kl.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Bytes of device workspace for a call with these sizes (chunk <= 0: the
 * default chunk).  Returns 0 for invalid sizes.  Per chunk of positions it
 * holds each row's largest key per 128-column vocabulary block
 * (8 * ceil(V / 128) bytes per row), the row's threshold, count and redo mark
 * (16 bytes) and its candidate list of up to 128 K entries (8 bytes each):
 * with the row's K-th largest block key as threshold the candidates all lie
 * in the K blocks whose largest key reaches it.
 */
size_t kd_topk_cache_workspace_bytes(int64_t N, int64_t d, int64_t V, int32_t K, int64_t chunk);

/* The chunk (positions per pass) used when a call passes chunk <= 0. */
int64_t kd_topk_cache_default_chunk(int64_t N, int64_t V, int32_t K);

/*
 * Writes the top-K cache of h against W.  Per chunk of positions: a
 * tensor-core pass computes z for the first max(K, V / 1024) blocks of 128
 * columns only and keeps each block's largest rank key; each row's threshold
 * is the K-th largest of those keys (at least K logits reach it, so no top-K
 * logit is below it); a second pass computes all of z with the same tiles
 * (bit-identical logits), keeps every block's largest key and collects every
 * key that reaches the threshold; a selection sorts each row's K best.  A row
 * whose candidates outgrow 128 K takes the K-th largest of all its block keys
 * as threshold instead and is collected again by a third pass, which does no
 * work when no row overflowed.
 * Errors: KD_ERR_INVALID_ARG (a NULL pointer, N < 0, d, V or K < 1, K > V),
 * KD_ERR_UNSUPPORTED (d % 8 != 0, K > KD_MAX_K, sizes beyond 2^31),
 * KD_ERR_WORKSPACE, KD_ERR_CUDA.  With N = 0 nothing is launched.
 */
kd_status kd_topk_cache_build(const void* h, const void* W, int64_t N, int64_t d, int64_t V,
                              int32_t K, int64_t chunk, int32_t* topk_idx, float* topk_logit,
                              void* workspace, size_t ws_bytes, uint32_t* dev_err_flags,
                              cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KD_TOPK_CACHE_H */
