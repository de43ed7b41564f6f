// kd_internal.h -- shared between the host driver and the kernel files of
// the kd_topk_kl library: tile constants, the workspace plan, and the launch
// functions of every kernel.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "kd_topk_kl.h"
#include "kd_topk_kl_steps.h"

namespace kd {

// Tensor-core tiles: a CTA pair owns a 256 x 256 output tile; each CTA holds
// its 128 rows x 256 fp32 columns in TMEM (two of them, double-buffered) and
// streams 64-deep K blocks of its halves of both operands.
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
// Largest default chunk, in tokens.
constexpr int64_t kMaxChunk = 8192;
// The chunk's hidden states are re-read by every tile of its GEMM launches,
// so the default chunk keeps them within this many bytes: on B300 about 60 MB
// of L2 serve re-reads (a buffer re-read by all SMs hits 98 % at 48 MB, 90 %
// at 64 MB, 25 % at 96 MB), and the streamed operand tiles need the rest.
constexpr int64_t kChunkL2Bytes = int64_t(48) << 20;
// Largest multiple of 128 rows (at least 128) whose `row_bytes` per row of
// hidden states fit in kChunkL2Bytes.
inline int64_t l2_chunk_cap(int64_t row_bytes) {
  const int64_t c = kChunkL2Bytes / (row_bytes < 1 ? 1 : row_bytes) / 128 * 128;
  return c < 128 ? 128 : c;
}
// The logsumexp statistics are kept per 128-column block of the vocabulary.
constexpr int kPB = 128;
// A sorted-index slot that holds no entry (dropped, or padding).
constexpr int kNoIndex = 0x7fffffff;

__host__ __device__ constexpr int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }
__host__ __device__ constexpr int64_t ceil_div(int64_t x, int64_t m) { return (x + m - 1) / m; }

// Host helpers shared by the entry points.
inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Streaming multiprocessors of the current device (0 on error).
inline int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// In host functions returning kd_status: a failed CUDA call returns
// KD_ERR_CUDA; KD_LAUNCH also brackets the launch with the optional timing
// events (needs a `stream` in scope).
#define KD_CUDA(x)                                    \
  do {                                                \
    if ((x) != cudaSuccess) return KD_ERR_CUDA;       \
  } while (0)
#define KD_LAUNCH(kind, x)                            \
  do {                                                \
    ::kd::TimedLaunch timed_launch_(kind, stream);    \
    KD_CUDA(x);                                       \
  } while (0)

// A named NVTX range around a library call or one chunk of it, visible to
// profilers that trace NVTX (ncu --nvtx); without one attached, the push and
// pop are no-ops.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Kernel kinds, for the optional per-launch timing (kd_timing_enable).
enum KernelKind {
  kTeacherPrep,
  kCompact,
  kZeroRows,
  kGatherRows,
  kBucketOffsets,
  kPass1Gemm,
  kLseCombine,
  kGradTile,
  kBwdGemm,
  kFinalize,
  kSimtPass1,
  kSimtGemm,
  kTopkBlockMax,
  kTopkThreshold,
  kTopkCandidates,
  kTopkSelect,
  kMaskRows,
  kFullPass1Gemm,
  kFullLseCombine,
  kFullGradTile,
  kTopkRefine,
  kTopkRedo,
  kGradPrepare,
  kNumKinds
};

// Brackets one kernel launch with CUDA events on its stream while timing is
// enabled (process-wide record guarded by a mutex; events of the current
// device).
struct TimedLaunch {
  TimedLaunch(int kind, cudaStream_t s);
  ~TimedLaunch();
  int kind;
  int dev = 0;
  cudaStream_t s;
  cudaEvent_t a = nullptr;
};

// Workspace plan for one call; all offsets 256-byte aligned.
struct Plan {
  int64_t N, d, V, K, chunk, cpad, n_pb, ldg, n_chunks;
  kd_dtype dtype;
  size_t elem;  // bytes per h/W/G element
  kd_workspace_layout lay;
};

// Fills `p` and returns KD_OK, or an error for invalid sizes.
kd_status make_plan(int64_t N, int64_t d, int64_t V, int32_t K, int64_t chunk, kd_dtype dtype,
                    Plan* p);
int64_t default_chunk(int64_t N, int64_t d, int64_t V, kd_dtype dtype);

// Control words at the start of the workspace.
struct Ctrl {
  uint32_t err;       // error flags when the caller passes none
  int32_t n_valid;    // number of valid rows
  double loss_sum;    // sum of the per-row loss terms
  int64_t n_valid64;  // the same count, the default normaliser of the loss
};

// Per-chunk pointers into the workspace that the row kernels use.
struct ChunkArgs {
  int64_t row0;          // first compacted row of this chunk
  int chunk;             // capacity of the chunk, in rows
  int64_t cpad;          // row stride of the per-chunk statistic arrays
  const int32_t* n_valid;  // valid rows of this call (compacted row count)
  const int64_t* n_norm;   // the loss's divisor: this call's count, or the
                           // count of the whole data-parallel batch
  const int32_t* rows;   // compacted row -> original row
  const int32_t* idx_sorted;
  const float* p_sorted;
  int K;
  int V;
  int n_pb;
  int64_t ldg;
  uint16_t* boff;        // [n_pb + 1][cpad] first sorted entry of each 128-column block
  float* part_m;         // [n_pb][cpad]  reference of block b's exponentials (then alpha_b)
  float* part_l;         // [n_pb][cpad]  block sum of 2^(s2 - reference)
  float* part_ps;        // [n_pb][cpad]  block sum of p_k * s2_k over teacher entries
  // One reference per row (bf16 path with gradients; nullptr otherwise),
  // indexed by the chunk's row i (the arrays start at the chunk's first row):
  float* mref;           // row i's reference m_i (log2 units): the student's
                         // logit at the teacher's most probable entry; after
                         // the logsumexp combine, the row's common reference M_i
  int32_t* row_flag;     // 1: some block of row i kept its own maximum
  float* alpha_row;      // 2^(M_i - lse2_i) / (T n): dL/dz = alpha_row * stored tile
  float* beta_row;       // 2^(lse2_i - M_i)
};

// A block of pass 1 stores its exponentials relative to the row's reference
// m_i when its own maximum is at most this far (log2 units) above m_i, so the
// stored values stay below 2^kRefSlack and the gradient products' fp32 sums
// far from overflow; otherwise relative to its own maximum (and the row is
// rescaled to one reference before the gradient products).
constexpr float kRefSlack = 40.f;

// ----------------------------------------------------------- row kernels
// top1 (optional, [N]): index of each valid row's most probable teacher entry.
cudaError_t launch_teacher_prep(const int32_t* idx, const float* logit, const uint8_t* mask,
                                int64_t N, int K, int64_t V, float T, int32_t* row_ok,
                                int32_t* idx_sorted, float* p_sorted, float* plogp, float* psum,
                                int32_t* top1, uint32_t* err, cudaStream_t s);
// Compacted valid-row map and the count (also copied to *n_valid_out, a
// device int64, when that is non-null).
cudaError_t launch_compact(const int32_t* row_ok, int64_t N, int32_t* rows, Ctrl* ctrl,
                           int64_t* n_valid_out, cudaStream_t s);
// With a.mref != nullptr (bf16), also the row references m_i = k2 * h_r . W[top1_r]
// and cleared row flags.
cudaError_t launch_gather_rows(const void* h, size_t elem, int64_t d, const ChunkArgs& a,
                               void* hc, const void* W, const int32_t* top1, float k2,
                               cudaStream_t s);
cudaError_t launch_bucket_offsets(const ChunkArgs& a, cudaStream_t s);
cudaError_t launch_lse(const ChunkArgs& a, const float* plogp, const float* psum, float T,
                       float* lse, float* loss_rows, cudaStream_t s);
cudaError_t launch_grad_tile(const ChunkArgs& a, void* g, size_t elem, float T, cudaStream_t s);
// bf16 path with one reference per row: prepares the stored exponentials u
// [cpad, ldg] and the gathered h [cpad, d] for the gradient products:
//   rows whose blocks kept their own maximum are rescaled to one reference;
//   u[i, v] -= (sum of p over row i's teacher entries at v) * beta_row[i];
//   hc[i, :] = alpha_row[i] * hc[i, :]  (bf16);
//   rows count .. round_up(count, 64) of u are zeroed.
// Then dL/dz = alpha_row * u, grad_h = alpha_row * (u W), grad_W = u^T hc.
cudaError_t launch_grad_prepare(const ChunkArgs& a, uint16_t* u, uint16_t* hc, int64_t d,
                                cudaStream_t s);
// loss = (sum of the valid rows' loss terms) / *n_norm (0 when *n_norm <= 0).
cudaError_t launch_finalize(const float* loss_rows, Ctrl* ctrl, const int64_t* n_norm,
                            float* loss, cudaStream_t s);
cudaError_t launch_zero_invalid_rows(const int32_t* row_ok, int64_t N, int64_t d, float* grad_h,
                                     cudaStream_t s);

// full-vocabulary loss
cudaError_t launch_mask_rows(const uint8_t* mask, int64_t N, int32_t* row_ok, cudaStream_t s);
cudaError_t launch_lse_dual(const ChunkArgs& a, float* part_mt, const float* part_lt,
                            const float* part_a, float T, float* lse, float* loss_rows,
                            cudaStream_t s);
cudaError_t launch_grad_tile_dual(const ChunkArgs& a, const float* alpha_t, const uint16_t* u_t,
                                  uint16_t* g, cudaStream_t s);

// ----------------------------------------------------------- fp32 CUDA-core path
cudaError_t launch_simt_pass1(const float* hc, const float* W, int64_t d, const ChunkArgs& a,
                              float k2, float* u, cudaStream_t s);
// C(m, n) (+)= sum_k A(m, k) B(k, n); A(m, k) = A[m * sam + k * sak], B(k, n) = B[k * sbk + n * sbn].
// M rows of C may be limited on the device to count = clamp(*n_valid - row0, 0, M_cap);
// with k_from_count the K extent is that count instead of Kfix.
struct SimtGemm {
  const float* A;
  int64_t sam, sak;
  const float* B;
  int64_t sbk, sbn;
  float* C;
  int64_t ldc;
  int64_t M_cap, N, Kfix;
  int m_from_count, k_from_count;
  const int32_t* row_map;  // C row = row_map[row_map_off + m] when non-null
  int64_t row_map_off;
  int accumulate;          // C += instead of C =; with K = 0 and accumulate = 0, C = 0
  const int32_t* n_valid;
  int64_t row0;
};
cudaError_t launch_simt_gemm(const SimtGemm& g, cudaStream_t s);

// ----------------------------------------------------------- tensor-core path
// Encodes a 2-D bf16 tensor map (inner dimension contiguous) with 128-byte
// swizzle and the given box.  Returns false if the driver rejects it.
bool encode_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                      uint64_t ld_elems, uint32_t box_inner, uint32_t box_outer);

// Tensor map of an output written by TMA stores from the 128-byte swizzle
// layout: fp32 (f32) or bf16 elements, [outer][inner] row-major with leading
// dimension ld_elems, one box = box_inner x box_outer (box_inner * element
// size = 128 bytes).
bool encode_tmap_store(CUtensorMap* m, const void* base, bool f32, uint64_t inner, uint64_t outer,
                       uint64_t ld_elems, uint32_t box_inner, uint32_t box_outer);

// An MN-major bf16 operand stored [outer = K][inner = MN] (MN contiguous,
// inner a multiple of 64), viewed as [inner / 64][outer][64] so that one box
// of `atoms` x box_k x 64 brings `atoms` consecutive 64-element atoms in the
// 128-byte swizzle layout.
bool encode_tmap_bf16_mn3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                           uint64_t ld_elems, uint32_t atoms, uint32_t box_k);

struct Pass1Args {
  const void* hc;  // [cpad, d] bf16
  const void* W;   // [V, d] bf16
  int64_t d;
  float k2;        // log2(e) / T
  bool row_ref;    // store u relative to the row references a.mref
  uint16_t* u;     // [cpad, ldg] bf16, written; nullptr: not stored (the loss alone)
  uint32_t* counter;
  uint32_t* err;
  int num_sms;
};
cudaError_t launch_tc_pass1(const Pass1Args& p, const ChunkArgs& a, cudaStream_t s);

// One or two GEMM problems in one persistent launch, fp32 results stored (or
// accumulated) row by row: out[row(m), n] (+)= sum_k A(m, k) B(n, k).
struct TcProblem {
  // Stored operands (bf16, row-major with the given leading dimension).  A
  // K-major operand is stored [rows, K] (inner = K); an MN-major one is
  // stored [K, rows] (inner = M or N).
  const void* A;
  int a_mn;
  int64_t a_inner, a_outer, lda;
  const void* B;
  int b_mn;
  int64_t b_inner, b_outer, ldb;
  int64_t M, N, K;   // output rows, output columns, reduction length (capacities)
  float* out;
  int64_t ldo;
  const float* row_scale;  // optional: output row m is multiplied by row_scale[m]
  const int32_t* row_map;  // output row = row_map[row_map_off + m] when non-null
  int64_t row_map_off;
  int accumulate;
  // With count_mode != 0 an extent is clamped on the device to
  // count = clamp(*n_valid - row0, 0, chunk):  1: M = count,  2: K = count.
  int count_mode;
};
struct TcGemmArgs {
  TcProblem pr[2];
  int nprob;
  const int32_t* n_valid;
  int64_t row0;
  int chunk;
  uint32_t* counter;
  uint32_t* err;
  int num_sms;
  uint64_t wait_limit_ns;  // 0: the default limit of every wait (4 s)
  int withhold_arrival;    // test of the bounded waits only (kd_umma_gemm_bf16_wait_test)
};
cudaError_t launch_tc_gemm(const TcGemmArgs& g, cudaStream_t s);

// The backward of one chunk in one launch: grad_h rows of the chunk = G_c W
// (stored through the compacted row map; row i multiplied by grad_h_scale[i]
// when given) and grad_W (+)= G_c^T h_c.
// G [cpad, ldg] bf16, W [V, d] bf16, hc [cpad, d] bf16.
cudaError_t launch_backward_gemms(const void* G, const void* W, const void* hc, int64_t d,
                                  int64_t V, int64_t cpad, int64_t ldg, int64_t chunk,
                                  const ChunkArgs& a, float* grad_h, float* grad_W,
                                  int accumulate, uint32_t* counter, uint32_t* err, int sms,
                                  cudaStream_t stream, const float* grad_h_scale = nullptr);

// Full-vocabulary loss, pass 1 over one chunk: teacher and student logits of
// each tile (problems 0 and 1 of one launch), their per-block statistics and
// stored exponentials.
struct DualPass1Args {
  const void* hc_t;  // [cpad, d_t] bf16, the chunk's teacher hidden states
  const void* W_t;   // [V, d_t] bf16
  const void* hc_s;  // [cpad, d_s] bf16
  const void* W_s;   // [V, d_s] bf16
  int64_t d_t, d_s;
  float k2;          // log2(e) / T
  uint16_t* u_t;     // [cpad, ldg] bf16, written
  uint16_t* u_s;     // [cpad, ldg] bf16, written
  float* part_mt;    // [n_pb][cpad]
  float* part_lt;
  float* part_a;
  uint32_t* counter;
  uint32_t* err;
  int num_sms;
};
cudaError_t launch_tc_dual_pass1(const DualPass1Args& p, const ChunkArgs& a, cudaStream_t s);

// Teacher top-K cache: the two tensor-core passes over one chunk of positions
// (z = h_c W^T).  pass 1 stores each 128-column block's largest rank key;
// pass 2 recomputes the same tiles and appends the keys that reach the row's
// threshold.
struct TopkGemmArgs {
  const void* h;      // [count, d] bf16, the chunk's first row
  const void* W;      // [V, d] bf16
  int64_t count, d, V;
  int64_t v_cols;     // logits computed: vocabulary columns [0, v_cols)
  const uint32_t* gate;  // optional: the launch does nothing while *gate == 0
  uint64_t* bkey;     // [count][ceil(V / 128)]
  const uint64_t* tau;
  uint32_t* cnt;
  uint64_t* cand;     // [count][cap]
  int64_t cap;
  uint32_t* counter;
  uint32_t* err;
  int num_sms;
};
cudaError_t launch_tc_topk(const TopkGemmArgs& g, int pass, cudaStream_t s);

}  // namespace kd
