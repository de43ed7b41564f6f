/*
 * kd_topk_kl.h -- fused chunked top-K KL distillation loss on B300 (sm_103a).
 *
 * The operation is the KL-divergence distillation loss of a student against an
 * offline teacher cache that keeps only the teacher's top K predictions per
 * position ("Efficient Knowledge Distillation for LLMs: Offline Top-K Logits
 * and a Fused Chunked KL Loss"; ai2day.live story, section "What did the
 * researchers change?": the teacher's top 100 predictions per position are
 * cached once, and the loss is computed over the sequence chunk by chunk, each
 * chunk calculated and discarded, the backward pass recomputing what it needs).
 * The loss is computed from the student's final hidden states and LM-head
 * weight without ever building the N x V student-logit grid (aiphreaks.com
 * summary, second paragraph; elseif.net summary, third paragraph); extra
 * device memory is O(chunk * V + N * K).
 *
 * Definitions (natural log; T is the temperature shared by teacher and student):
 *   p_r      = softmax over the K cached entries of (topk_logit_r / T)
 *   z        = h W^T,   s = z / T,   lse_r = logsumexp over the vocabulary of s_r
 *   loss     = (1 / N_valid) * sum over valid rows r of
 *                sum_k p_rk * (log p_rk - (s_{r, idx_rk} - lse_r))
 *   dL/dz_rv = (softmax(s_r)_v - sum_{k : idx_rk = v} p_rk) / (T * N_valid)
 *   grad_h   = (dL/dz) W        grad_W = (dL/dz)^T h
 * There is no T^2 factor.  N_valid counts the valid rows; with N_valid = 0 the
 * loss and both gradients are 0.
 *
 * Layouts (all row-major, contiguous, 16-byte aligned device buffers):
 *   h          [N, d]   bf16 or fp32 (dtype)          student final hidden states
 *   W          [V, d]   same dtype as h                LM-head weight (nn.Linear layout)
 *   topk_idx   [N, K]   int32                          teacher vocabulary indices
 *   topk_logit [N, K]   fp32                           teacher logits (or log-probs)
 *   mask       [N]      uint8, 1 = valid, 0 = ignored; NULL means every row valid
 *   loss       [1]      fp32, written
 *   grad_h     [N, d]   fp32, overwritten (rows that are not valid are set to 0)
 *   grad_W     [V, d]   fp32, overwritten
 * d must be a multiple of 8 (bf16) or 4 (fp32): the rows are read by the tensor
 * memory accelerator, whose strides are multiples of 16 bytes.
 *
 * Row validity and data errors (found on the device, reported through
 * *dev_err_flags, which the library ORs bits into; the caller zeroes it and
 * reads it after synchronising the stream):
 *   KD_FLAG_INDEX_RANGE  an index of a valid row lies outside [0, V): that
 *                        entry is dropped from the teacher distribution (as if
 *                        its logit were -inf).
 *   KD_FLAG_BAD_TEACHER  a valid row whose in-range teacher logits contain NaN
 *                        or +inf, or no finite value: the row is treated as
 *                        masked (no loss, zero grad_h row, not in N_valid).
 *   KD_FLAG_TIMEOUT      a wait inside a kernel gave up after its time limit;
 *                        the results of that call are not valid.
 * A -inf teacher logit is legal and gives that entry probability 0.  A
 * duplicate index within a row adds its probabilities.  Masked rows' data
 * (h, topk_idx, topk_logit) is never read for a result.
 *
 * Ownership and execution: the caller owns every buffer (inputs, outputs and
 * the workspace).  The library allocates no memory and keeps no per-call state;
 * every call is stream-ordered and asynchronous on `stream` (0 = the legacy
 * default stream).  The returned status reports only the synchronous host-side
 * checks and launch errors.  Two calls may run concurrently only with distinct
 * workspaces.
 */
#ifndef KD_TOPK_KL_H
#define KD_TOPK_KL_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KD_OK = 0,
  KD_ERR_INVALID_ARG = 1,  /* null pointer, negative size, K < 1, bad T, ... */
  KD_ERR_UNSUPPORTED = 2,  /* a size this build does not handle (see below)  */
  KD_ERR_WORKSPACE = 3,    /* workspace NULL or smaller than required        */
  KD_ERR_CUDA = 4          /* a CUDA call or kernel launch failed            */
} kd_status;

typedef enum { KD_BF16 = 0, KD_FP32 = 1 } kd_dtype;

#define KD_FLAG_INDEX_RANGE 1u
#define KD_FLAG_BAD_TEACHER 2u
#define KD_FLAG_TIMEOUT 4u
/* A bound the kernels rely on was found violated (a defect, not a data
 * error); the results of the call are not valid. */
#define KD_FLAG_INTERNAL 8u

/* Largest K accepted (the per-row sort of the teacher entries runs in shared
 * memory); larger K returns KD_ERR_UNSUPPORTED. */
#define KD_MAX_K 4096

/*
 * Bytes of device workspace a call with these sizes needs.  chunk <= 0 asks
 * for the default chunk (kd_topk_kl_default_chunk).  Returns 0 for invalid
 * sizes.  The workspace holds, per call: the teacher probabilities and sorted
 * indices (O(N K)), per-row statistics (O(N)), and one chunk's
 * vocabulary-wide buffers (O(chunk V)).  It needs no initialisation.
 */
size_t kd_topk_kl_workspace_bytes(int64_t N, int64_t d, int64_t V, int32_t K, int64_t chunk,
                                  kd_dtype dtype);

/*
 * Bytes of workspace kd_topk_kl_fwd (the loss alone) needs: the same layout
 * without the chunk's vocabulary-wide exponential tile, which only the
 * gradients use -- O(N K + chunk V / 64) instead of O(N K + chunk V).  A
 * workspace of kd_topk_kl_workspace_bytes serves both calls.  Returns 0 for
 * invalid sizes.
 */
size_t kd_topk_kl_fwd_workspace_bytes(int64_t N, int64_t d, int64_t V, int32_t K, int64_t chunk,
                                      kd_dtype dtype);

/*
 * The chunk (in tokens) used when a call passes chunk <= 0: equal chunks of a
 * multiple of 128 tokens, at most 8192, small enough that the chunk's
 * vocabulary buffer stays near 4 GiB and its hidden states (chunk x d
 * elements) within 48 MiB, the part of L2 that holds data re-read by every
 * tile of the chunk's GEMMs.
 */
int64_t kd_topk_kl_default_chunk(int64_t N, int64_t d, int64_t V, kd_dtype dtype);

/*
 * Loss, grad_h and grad_W in one pass over the token chunks.
 *   chunk      tokens per chunk (the unit whose vocabulary-wide buffers live
 *              in the workspace); <= 0 picks the default.  The result does not
 *              depend on it beyond floating-point rounding.
 *   T          temperature, finite and > 0.
 *   dev_err_flags  optional device uint32 (see above); NULL keeps the flags in
 *              the workspace only.
 * Errors: KD_ERR_INVALID_ARG (a required pointer is NULL; N < 0; d, V or K < 1;
 * K > KD_MAX_K is KD_ERR_UNSUPPORTED; T not finite or <= 0), KD_ERR_UNSUPPORTED
 * (d not a multiple of 8 for bf16 / 4 for fp32), KD_ERR_WORKSPACE, KD_ERR_CUDA.
 * With N = 0, h, topk_idx, topk_logit, mask and grad_h may be NULL; loss and
 * grad_W are written as 0.
 */
kd_status kd_topk_kl_fwd_bwd(const void* h, const void* W, kd_dtype dtype,
                             const int32_t* topk_idx, const float* topk_logit,
                             const uint8_t* mask, int64_t N, int64_t d, int64_t V, int32_t K,
                             float T, int64_t chunk, float* loss, float* grad_h, float* grad_W,
                             void* workspace, size_t ws_bytes, uint32_t* dev_err_flags,
                             cudaStream_t stream);

/* The loss alone (same definition and arguments, no gradient outputs); its
 * workspace need only be kd_topk_kl_fwd_workspace_bytes long. */
kd_status kd_topk_kl_fwd(const void* h, const void* W, kd_dtype dtype, const int32_t* topk_idx,
                         const float* topk_logit, const uint8_t* mask, int64_t N, int64_t d,
                         int64_t V, int32_t K, float T, int64_t chunk, float* loss,
                         void* workspace, size_t ws_bytes, uint32_t* dev_err_flags,
                         cudaStream_t stream);

/*
 * Data parallelism: one batch split over several ranks (processes, one GPU
 * each).  Every rank owns some of the tokens and their teacher-cache rows; W
 * is replicated.  The loss of the batch is the mean over ALL its valid tokens
 * (the token-level mean above, taken over the whole batch), so each rank's
 * terms must be divided by N_valid of the whole batch, which is known only
 * once every rank has counted its own valid rows.  Two calls split
 * kd_topk_kl_fwd_bwd at that point:
 *   1. kd_topk_kl_prepare     teacher preparation and the valid-row map of
 *                             this rank's tokens; writes this rank's N_valid
 *                             to *n_valid (device int64, optional);
 *   2. (caller)               sums n_valid over the ranks (an all-reduce on
 *                             the same stream: no host synchronisation);
 *   3. kd_topk_kl_fwd_bwd_prepared / kd_topk_kl_fwd_prepared
 *                             the chunk loop over the prepared workspace with
 *                             the divisor *n_norm (device int64): loss =
 *                             (sum of this rank's loss terms) / n_norm, and
 *                             dL/dz = (softmax - p scattered) / (T n_norm).
 * Summing loss and grad_W over the ranks then gives the batch's loss and
 * grad_W exactly as one call over the whole batch would; grad_h rows stay
 * with their rank.  kd_topk_kl_fwd_bwd is step 1 followed by step 3 with
 * n_norm = this rank's own count.
 *
 * The prepared call must use the same sizes (N, d, V, K, chunk, dtype), T and
 * workspace as the kd_topk_kl_prepare call, be ordered after it (same stream,
 * or an event), and no other call may use that workspace in between.
 * n_norm == NULL divides by this rank's own count; *n_norm <= 0 gives a zero
 * loss and zero gradients (no valid token in the whole batch); *n_norm
 * smaller than this rank's count is a caller error (the results are scaled
 * accordingly, nothing is checked).  The prepare call needs a workspace of at
 * least kd_topk_kl_fwd_workspace_bytes; kd_topk_kl_fwd_bwd_prepared needs
 * kd_topk_kl_workspace_bytes.  Errors as for kd_topk_kl_fwd_bwd; the data
 * flags (INDEX_RANGE, BAD_TEACHER) are raised by the prepare call.
 */
kd_status kd_topk_kl_prepare(const int32_t* topk_idx, const float* topk_logit,
                             const uint8_t* mask, int64_t N, int64_t d, int64_t V, int32_t K,
                             float T, int64_t chunk, kd_dtype dtype, void* workspace,
                             size_t ws_bytes, int64_t* n_valid, uint32_t* dev_err_flags,
                             cudaStream_t stream);

kd_status kd_topk_kl_fwd_bwd_prepared(const void* h, const void* W, kd_dtype dtype, int64_t N,
                                      int64_t d, int64_t V, int32_t K, float T, int64_t chunk,
                                      const int64_t* n_norm, float* loss, float* grad_h,
                                      float* grad_W, void* workspace, size_t ws_bytes,
                                      uint32_t* dev_err_flags, cudaStream_t stream);

kd_status kd_topk_kl_fwd_prepared(const void* h, const void* W, kd_dtype dtype, int64_t N,
                                  int64_t d, int64_t V, int32_t K, float T, int64_t chunk,
                                  const int64_t* n_norm, float* loss, void* workspace,
                                  size_t ws_bytes, uint32_t* dev_err_flags, cudaStream_t stream);

/*
 * kd_topk_kl_fwd_bwd_noalloc -- kd_topk_kl_fwd_bwd for callers that cannot
 * allocate device memory.  (The write-ups have no counterpart: this is an
 * interface convenience, not part of the method.)
 *
 * Who needs it: code that may not call cudaMalloc -- a process whose memory
 * pool owns the device and forbids allocations beside it, a plug-in that is
 * handed device pointers for its inputs and outputs but no allocator -- still
 * has to supply the workspace that kd_topk_kl_fwd_bwd takes.  This call uses instead a scratch array of
 * KD_NOALLOC_SCRATCH_BYTES that the library holds in device memory: every GPU
 * that loads the library keeps that array until the process exits.  The call
 * itself allocates nothing (no cudaMalloc, cudaFree or allocating library
 * routine).
 *
 * Arguments, results, device error flags and host-side errors are those of
 * kd_topk_kl_fwd_bwd, without the workspace.  chunk <= 0 picks the largest
 * chunk (a multiple of 128 tokens, at most kd_topk_kl_default_chunk) whose
 * workspace fits in the array; a request whose workspace
 * (kd_topk_kl_workspace_bytes) exceeds KD_NOALLOC_SCRATCH_BYTES even at that
 * smallest chunk, or at the chunk the caller passed, returns KD_ERR_WORKSPACE
 * before any CUDA call.
 *
 * Set-up: the first call on a device, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress, which may load the library's
 * device code); make that first call before any stream capture.  Every call
 * on a device shares the one array, and the array keeps the previous call's
 * contents (each call clears the parts that must start at zero).  Calls that
 * overlap on the GPU -- on different streams, or from different host threads
 * -- race on the array and give wrong results: order them on one stream.
 */
#define KD_NOALLOC_SCRATCH_BYTES (64u << 20)

kd_status kd_topk_kl_fwd_bwd_noalloc(const void* h, const void* W, kd_dtype dtype,
                                     const int32_t* topk_idx, const float* topk_logit,
                                     const uint8_t* mask, int64_t N, int64_t d, int64_t V,
                                     int32_t K, float T, int64_t chunk, float* loss,
                                     float* grad_h, float* grad_W, uint32_t* dev_err_flags,
                                     cudaStream_t stream);

/* A static, human-readable name for a status code. */
const char* kd_status_string(kd_status status);

#ifdef __cplusplus
}
#endif

#endif /* KD_TOPK_KL_H */
