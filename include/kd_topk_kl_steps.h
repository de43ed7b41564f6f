/*
 * kd_topk_kl_steps.h -- step-level entry points of the kd_topk_kl library.
 *
 * These expose pieces of the fused top-K KL loss (see kd_topk_kl.h) so that a
 * test can check each one on its own:
 *   - the layout of the workspace, so the per-row intermediate results a call
 *     leaves there (the student log-partition lse_r and the per-row loss terms
 *     of "Efficient Knowledge Distillation for LLMs: Offline Top-K Logits and a
 *     Fused Chunked KL Loss", ai2day.live story, "What did the researchers
 *     change?") can be compared with a reference;
 *   - the tensor-core matrix product the three contractions of that loss use
 *     (z = h W^T, grad_h = G W, grad_W = G^T h), as a plain GEMM.
 * Same conventions as kd_topk_kl.h: caller-owned device buffers, nothing
 * allocated, stream-ordered, host-side status only.
 */
#ifndef KD_TOPK_KL_STEPS_H
#define KD_TOPK_KL_STEPS_H

#include "kd_topk_kl.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Where a call with these sizes keeps its intermediates inside the workspace
 * (byte offsets from the workspace base, each 256-byte aligned).  Valid after
 * a kd_topk_kl_fwd_bwd / kd_topk_kl_fwd call has completed on its stream:
 *   ctrl:       uint32 error flags at +0, int32 N_valid at +4, double loss sum at +8,
 *               int64 N_valid at +16
 *   rows:       int32 [N]  original row of the i-th valid row (i < N_valid)
 *   lse:        fp32  [N]  lse_i of the i-th valid row (natural log, of s = z/T)
 *   loss_rows:  fp32  [N]  loss term of the i-th valid row (before the 1/N_valid)
 * Teacher preparation, for every valid original row r:
 *   idx_sorted: int32 [N, K]  row r's in-range teacher indices in increasing
 *                             order (equal indices in any order), then
 *                             0x7fffffff up to K entries
 *   p_sorted:   fp32  [N, K]  the teacher probability of each of those entries
 *                             (softmax of logit / T over the row's in-range
 *                             entries), 0 for the padding
 *   plogp:      fp32  [N]     sum of p ln p over row r's entries
 *   psum:       fp32  [N]     sum of p over row r's entries (1 up to rounding)
 *   top1:       int32 [N]     index of row r's most probable entry (the lower
 *                             index among equal probabilities)
 * The last chunk that holds valid rows, j = (N_valid - 1) / chunk, with
 * count = N_valid - j * chunk rows; its i-th row (i < count) is the original
 * row rows[j * chunk + i]:
 *   boff:       uint16 [n_pb + 1, chunk_pad]  boff[b][i] = position in that
 *                             row's sorted entries of the first one whose
 *                             index is >= 128 b
 *   g:          [chunk_pad, ld_g], after kd_topk_kl_fwd_bwd only: the
 *               gradient of the loss with respect to the student logits,
 *               dL/dz[i, v] = (softmax(s_i)_v - sum of p over the row's entries
 *               with index v) / (T N_valid), for v < V:
 *                 KD_FP32: dL/dz itself (fp32); columns V .. ld_g - 1 zero;
 *                 KD_BF16: bf16 values g' with dL/dz[i, v] = alpha_i * g'[i, v]
 *                          (alpha_i in rowstat below): the row's exponentials
 *                          relative to one reference, minus the teacher's
 *                          probabilities scaled to match
 *   rowstat:    fp32 [4, N] (KD_BF16 with gradients), for the i-th valid row
 *               of the call (every chunk, compacted order): [0] the common
 *               reference M_i (log2 units) of its stored values, [1] (int32) 1
 *               if some vocabulary block kept its own maximum as reference (the
 *               row was then rescaled to M_i), [2] alpha_i, [3] 1 / (alpha_i T
 *               N_valid); alpha_i of the last chunk's row i is at
 *               [2, j * chunk + i]; part_m holds each block's reference
 *   hc:         [chunk_pad, d] the chunk's rows of h (KD_BF16 with gradients:
 *               multiplied by alpha_i and rounded to bf16, so that grad_W
 *               receives g'^T hc)
 * The other regions, and the rows of boff and g beyond count, are scratch
 * space whose contents are not specified.
 */
typedef struct {
  int64_t chunk;      /* resolved chunk, in tokens                              */
  int64_t chunk_pad;  /* rows of each per-chunk buffer (multiple of 128)        */
  int64_t n_pb;       /* 128-column vocabulary blocks, ceil(V / 128)           */
  int64_t ld_g;       /* row stride, in elements, of the per-chunk vocab buffer */
  size_t off_ctrl;
  size_t off_row_ok;
  size_t off_rows;
  size_t off_idx_sorted;
  size_t off_p_sorted;
  size_t off_plogp;
  size_t off_psum;
  size_t off_lse;
  size_t off_loss_rows;
  size_t off_part_m;
  size_t off_part_l;
  size_t off_part_ps;
  size_t off_boff;
  size_t off_top1;
  size_t off_rowstat;
  size_t off_hc;
  size_t off_g;
  size_t off_sched;
  size_t total;
} kd_workspace_layout;

kd_status kd_topk_kl_workspace_layout(int64_t N, int64_t d, int64_t V, int32_t K, int64_t chunk,
                                      kd_dtype dtype, kd_workspace_layout* out);

/*
 * The same layout for a kd_full_kl_fwd_bwd call (kd_full_kl.h): ctrl, rows,
 * lse (of the student's s) and loss_rows as above, and g (bf16), the last
 * chunk's gradient with respect to the student logits, (softmax(s_i)_v -
 * softmax(t_i)_v) / (T N_valid), in the same rows and columns as above; the
 * regions that belong to the top-K cache (sorted teacher entries, plogp,
 * psum, part_ps, boff) do not exist there and are reported as offset 0.
 */
kd_status kd_full_kl_workspace_layout(int64_t N, int64_t d_s, int64_t d_t, int64_t V,
                                      int64_t chunk, kd_workspace_layout* out);

/*
 * D[M, N] (fp32, row-major, leading dimension N) = sum_k A(m, k) * B(n, k) on
 * the tcgen05 tensor cores, bf16 inputs, fp32 accumulation; D += ... when
 * accumulate != 0.
 *   a_mn_major = 0: A is [M, K] row-major (K contiguous); 1: A is [K, M] (M contiguous)
 *   b_mn_major = 0: B is [N, K] row-major (K contiguous); 1: B is [K, N] (N contiguous)
 * The contiguous dimension of each operand must be a multiple of 8 elements
 * (16-byte rows).  counter is one device uint32 of scratch that the call
 * resets and uses to hand out tiles.  Errors as in kd_topk_kl.h.
 */
kd_status kd_umma_gemm_bf16(const void* A, const void* B, float* D, int64_t M, int64_t N,
                            int64_t K, int a_mn_major, int b_mn_major, int accumulate,
                            uint32_t* counter, uint32_t* dev_err_flags, cudaStream_t stream);

/*
 * Test of the time-bounded waits (the write-ups define no counterpart).  Runs
 * the kd_umma_gemm_bf16 kernel (A [M, K], B [N, K], both K-major) with one
 * barrier arrival deliberately never made: the first operand stage of the
 * first tile is never announced, so the MMA's wait for it cannot complete.
 * Every wait of the kernel is limited to wait_limit_us microseconds; the wait
 * that runs out raises KD_FLAG_TIMEOUT in *dev_err_flags, tells every other
 * role of both CTAs of the pair to stop, lets in-flight copies and MMAs
 * finish, frees the tensor memory and returns -- the context stays usable.
 * D is left partly written.  Nothing faults or hangs: the call shows that a
 * protocol error ends the kernel with a status the host can read.
 */
kd_status kd_umma_gemm_bf16_wait_test(const void* A, const void* B, float* D, int64_t M,
                                      int64_t N, int64_t K, uint32_t wait_limit_us,
                                      uint32_t* counter, uint32_t* dev_err_flags,
                                      cudaStream_t stream);

/*
 * Kernel timing (instrumentation; the write-ups define no counterpart).  While
 * enabled, the library brackets each of its kernel launches with a pair of
 * CUDA events recorded on the launching stream.  kd_timing_collect waits for
 * those events, returns one entry per kernel kind (launch count and summed
 * device time), and clears the record.  One record for the whole process,
 * guarded by a lock: calls from several host threads and on several devices
 * may record at the same time (each event is made on the device of the
 * stream it brackets); collect returns them all together.  Off by default.
 */
typedef struct {
  char name[32];      /* kernel kind, e.g. "pass1_gemm", "bwd_gemm"          */
  int64_t launches;   /* launches recorded since the last collect             */
  double total_ms;    /* summed CUDA-event time of those launches             */
} kd_timing_entry;

kd_status kd_timing_enable(int on);
/* Writes up to max_entries entries; *n_entries receives the number of kinds. */
kd_status kd_timing_collect(kd_timing_entry* out, int32_t max_entries, int32_t* n_entries);

#ifdef __cplusplus
}
#endif

#endif /* KD_TOPK_KL_STEPS_H */
