// kd_api.cu -- host side of the kd_topk_kl C ABI: argument checks, the
// workspace plan, tensor-map encoding and the chunk loop that launches the
// kernels of the fused top-K KL loss on the caller's stream.
//
// The chunk loop is the method of "Efficient Knowledge Distillation for LLMs:
// Offline Top-K Logits and a Fused Chunked KL Loss" (ai2day.live story, "What
// did the researchers change?"): the sequence is sliced into chunks, each
// chunk's vocabulary-wide buffers are computed, used and overwritten by the
// next chunk, so device memory grows as O(chunk * V + N * K), never O(N * V).
#include <math.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "kd_internal.h"

namespace kd {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// ------------------------------------------------------------- kernel timing
const char* const kKindNames[kNumKinds] = {
    "teacher_prep", "compact",    "zero_invalid_rows", "gather_rows", "bucket_offsets",
    "pass1_gemm",   "lse_combine", "grad_tile",        "bwd_gemm",    "finalize",
    "simt_pass1",   "simt_gemm",   "topk_block_max",   "topk_threshold",
    "topk_candidates", "topk_select", "mask_rows", "full_pass1_gemm", "full_lse_combine",
    "full_grad_tile", "topk_refine", "topk_redo", "grad_prepare"};

// Timing records and spare events.  An event belongs to the device that was
// current when it was created and can be recorded only on that device's
// streams, so the spare events are kept per device; one mutex guards all of
// this state, so calls from several host threads may record concurrently.
struct TimingRec {
  int kind;
  int dev;
  cudaEvent_t a, b;
};
std::mutex g_timing_mu;
bool g_timing_on = false;
std::vector<TimingRec> g_recs;
std::vector<std::vector<cudaEvent_t>> g_event_pool;  // [device] spare events

// A spare event of device `dev` (created there when none is left); the
// caller holds g_timing_mu and `dev` is current.
cudaEvent_t pooled_event(int dev) {
  if (static_cast<int>(g_event_pool.size()) <= dev) g_event_pool.resize(dev + 1);
  std::vector<cudaEvent_t>& pool = g_event_pool[dev];
  if (!pool.empty()) {
    cudaEvent_t e = pool.back();
    pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

TimedLaunch::TimedLaunch(int k, cudaStream_t st) : kind(k), s(st) {
  std::lock_guard<std::mutex> lock(g_timing_mu);
  if (!g_timing_on || cudaGetDevice(&dev) != cudaSuccess) return;
  a = pooled_event(dev);
  if (a != nullptr) cudaEventRecord(a, s);
}

TimedLaunch::~TimedLaunch() {
  if (a == nullptr) return;
  std::lock_guard<std::mutex> lock(g_timing_mu);
  cudaEvent_t b = pooled_event(dev);
  if (b == nullptr) {
    g_event_pool[dev].push_back(a);
    return;
  }
  cudaEventRecord(b, s);
  g_recs.push_back(TimingRec{kind, dev, a, b});
}

bool encode_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                      uint64_t ld_elems, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {ld_elems * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_store(CUtensorMap* m, const void* base, bool f32, uint64_t inner, uint64_t outer,
                       uint64_t ld_elems, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const uint64_t es = f32 ? 4 : 2;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {ld_elems * es};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_bf16_mn3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                           uint64_t ld_elems, uint32_t atoms, uint32_t box_k) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || inner % 64 != 0) return false;
  // [inner / 64][outer][64]: element (mn, k) at mn % 64 + k * ld + (mn / 64) * 64
  const cuuint64_t dims[3] = {64, outer, inner / 64};
  const cuuint64_t strides[2] = {ld_elems * 2, 128};
  const cuuint32_t box[3] = {64, box_k, atoms};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int64_t default_chunk(int64_t N, int64_t d, int64_t V, kd_dtype dtype) {
  const int64_t elem = dtype == KD_BF16 ? 2 : 4;
  const int64_t ldg = round_up(V, kBN);
  // Keep the per-chunk vocabulary buffer near 4 GiB: a few chunks per call
  // amortise the grad_W read-modify-write while the extra memory stays small
  // next to HBM.
  // The chunks are then made equal (multiples of 128 rows) so the last one
  // is not a small remainder.
  const int64_t budget = int64_t(4) << 30;
  int64_t cmax = budget / (ldg * elem);
  cmax = cmax / kBM * kBM;
  if (cmax < kBM) cmax = kBM;
  // The chunk's hidden states must stay resident in L2 (measured at 32K
  // tokens, d = 4096: chunk 8192 87.3 ms per step, 6144 85.3, 5120 84.6; at
  // d = 2880, 11008 tokens were 1.8 % slower than 8192).
  if (cmax > kMaxChunk) cmax = kMaxChunk;
  const int64_t cl2 = l2_chunk_cap(d * elem);
  if (cmax > cl2) cmax = cl2;
  const int64_t n = N < 1 ? 1 : N;
  const int64_t pieces = ceil_div(n, cmax);
  return round_up(ceil_div(n, pieces), kBM);
}

kd_status make_plan(int64_t N, int64_t d, int64_t V, int32_t K, int64_t chunk, kd_dtype dtype,
                    Plan* p) {
  if (dtype != KD_BF16 && dtype != KD_FP32) return KD_ERR_INVALID_ARG;
  if (N < 0 || d < 1 || V < 1 || K < 1) return KD_ERR_INVALID_ARG;
  if (K > KD_MAX_K) return KD_ERR_UNSUPPORTED;
  if (N >= (int64_t(1) << 31) || V >= (int64_t(1) << 31) - 1024 || d >= (int64_t(1) << 24))
    return KD_ERR_UNSUPPORTED;
  if ((dtype == KD_BF16 && d % 8 != 0) || (dtype == KD_FP32 && d % 4 != 0))
    return KD_ERR_UNSUPPORTED;
  Plan& P = *p;
  P.N = N;
  P.d = d;
  P.V = V;
  P.K = K;
  P.dtype = dtype;
  P.elem = dtype == KD_BF16 ? 2 : 4;
  int64_t c = chunk > 0 ? chunk : default_chunk(N, d, V, dtype);
  if (N > 0 && c > N) c = N;
  if (c < 1) c = 1;
  if (c >= (int64_t(1) << 30)) return KD_ERR_UNSUPPORTED;
  P.chunk = c;
  P.cpad = round_up(c, kBM);
  P.n_pb = ceil_div(V, kPB);
  P.ldg = round_up(V, kBN);
  P.n_chunks = N > 0 ? ceil_div(N, c) : 0;
  kd_workspace_layout& L = P.lay;
  memset(&L, 0, sizeof(L));
  L.chunk = P.chunk;
  L.chunk_pad = P.cpad;
  L.n_pb = P.n_pb;
  L.ld_g = P.ldg;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  const size_t n = static_cast<size_t>(N);
  const size_t nk = n * static_cast<size_t>(K);
  const size_t part = static_cast<size_t>(P.n_pb) * static_cast<size_t>(P.cpad);
  L.off_ctrl = take(256);
  L.off_row_ok = take(4 * n);
  L.off_rows = take(4 * n);
  L.off_idx_sorted = take(4 * nk);
  L.off_p_sorted = take(4 * nk);
  L.off_top1 = take(4 * n);
  L.off_plogp = take(4 * n);
  L.off_psum = take(4 * n);
  L.off_lse = take(4 * n);
  L.off_loss_rows = take(4 * n);
  L.off_part_m = take(4 * part);
  L.off_part_l = take(4 * part);
  L.off_part_ps = take(4 * part);
  L.off_boff = take(2 * (static_cast<size_t>(P.n_pb) + 1) * static_cast<size_t>(P.cpad));
  L.off_rowstat = take(4 * 4 * n);
  L.off_hc = take(static_cast<size_t>(P.cpad) * static_cast<size_t>(d) * P.elem);
  L.off_sched = take(256);
  // last: the loss alone stops here (kd_topk_kl_fwd_workspace_bytes)
  L.off_g = take(static_cast<size_t>(P.cpad) * static_cast<size_t>(P.ldg) * P.elem);
  L.total = o;
  return KD_OK;
}

cudaError_t launch_backward_gemms(const void* G, const void* W, const void* hc, int64_t d,
                                  int64_t V, int64_t cpad, int64_t ldg, int64_t chunk,
                                  const ChunkArgs& a, float* grad_h, float* grad_W,
                                  int accumulate, uint32_t* counter, uint32_t* err, int sms,
                                  cudaStream_t stream, const float* grad_h_scale) {
  TcGemmArgs g;
  memset(&g, 0, sizeof(g));
  TcProblem& gh = g.pr[0];  // grad_h rows of the chunk = G_c W
  gh.A = G;
  gh.a_mn = 0;
  gh.a_inner = V;
  gh.a_outer = cpad;
  gh.lda = ldg;
  gh.B = W;
  gh.b_mn = 1;
  gh.b_inner = d;
  gh.b_outer = V;
  gh.ldb = d;
  gh.M = chunk;
  gh.N = d;
  gh.K = V;
  gh.out = grad_h;
  gh.ldo = d;
  gh.row_map = a.rows;
  gh.row_map_off = a.row0;
  gh.row_scale = grad_h_scale;
  gh.accumulate = 0;
  gh.count_mode = 1;
  TcProblem& gw = g.pr[1];  // grad_W (+)= G_c^T h_c
  gw.A = G;
  gw.a_mn = 1;
  // G's columns V .. ldg are zero, so whole 64-column atoms may be read
  gw.a_inner = round_up(V, 64);
  gw.a_outer = cpad;
  gw.lda = ldg;
  gw.B = hc;
  gw.b_mn = 1;
  gw.b_inner = d;
  gw.b_outer = cpad;
  gw.ldb = d;
  gw.M = V;
  gw.N = d;
  gw.K = chunk;
  gw.out = grad_W;
  gw.ldo = d;
  gw.row_map = nullptr;
  gw.accumulate = accumulate;
  gw.count_mode = 2;
  g.nprob = 2;
  g.n_valid = a.n_valid;
  g.row0 = a.row0;
  g.chunk = a.chunk;
  g.counter = counter;
  g.err = err;
  g.num_sms = sms;
  return launch_tc_gemm(g, stream);
}

namespace {

struct Views {
  Ctrl* ctrl;
  int32_t* row_ok;
  int32_t* rows;
  int32_t* idx_sorted;
  float* p_sorted;
  float* plogp;
  float* psum;
  float* lse;
  float* loss_rows;
  float* part_m;
  float* part_l;
  float* part_ps;
  uint16_t* boff;
  int32_t* top1;
  float* mref;
  int32_t* row_flag;
  float* alpha_row;
  float* beta_row;
  void* hc;
  void* g;
  uint32_t* sched;
};

Views views(const Plan& P, void* ws) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  const kd_workspace_layout& L = P.lay;
  Views v;
  v.ctrl = reinterpret_cast<Ctrl*>(b + L.off_ctrl);
  v.row_ok = reinterpret_cast<int32_t*>(b + L.off_row_ok);
  v.rows = reinterpret_cast<int32_t*>(b + L.off_rows);
  v.idx_sorted = reinterpret_cast<int32_t*>(b + L.off_idx_sorted);
  v.p_sorted = reinterpret_cast<float*>(b + L.off_p_sorted);
  v.plogp = reinterpret_cast<float*>(b + L.off_plogp);
  v.psum = reinterpret_cast<float*>(b + L.off_psum);
  v.lse = reinterpret_cast<float*>(b + L.off_lse);
  v.loss_rows = reinterpret_cast<float*>(b + L.off_loss_rows);
  v.part_m = reinterpret_cast<float*>(b + L.off_part_m);
  v.part_l = reinterpret_cast<float*>(b + L.off_part_l);
  v.part_ps = reinterpret_cast<float*>(b + L.off_part_ps);
  v.boff = reinterpret_cast<uint16_t*>(b + L.off_boff);
  v.top1 = reinterpret_cast<int32_t*>(b + L.off_top1);
  float* rs = reinterpret_cast<float*>(b + L.off_rowstat);
  v.mref = rs;
  v.row_flag = reinterpret_cast<int32_t*>(rs + P.N);
  v.alpha_row = rs + 2 * P.N;
  v.beta_row = rs + 3 * P.N;
  v.hc = b + L.off_hc;
  v.g = b + L.off_g;
  v.sched = reinterpret_cast<uint32_t*>(b + L.off_sched);
  return v;
}

// Host-side checks of the sizes, the workspace and the stream's device; fills
// the plan.  `need_grads`: the workspace must hold the exponential tile.
kd_status check_call(int64_t N, int64_t d, int64_t V, int32_t K, float T, int64_t chunk,
                     kd_dtype dtype, bool need_grads, const void* workspace, size_t ws_bytes,
                     Plan* P) {
  kd_status st = make_plan(N, d, V, K, chunk, dtype, P);
  if (st != KD_OK) return st;
  if (!(T > 0.f) || !isfinite(T)) return KD_ERR_INVALID_ARG;
  // the loss alone never touches the last region (the chunk's exponential tile)
  const size_t need = need_grads ? P->lay.total : P->lay.off_g;
  if (workspace == nullptr || ws_bytes < need) return KD_ERR_WORKSPACE;
  if (!aligned16(workspace)) return KD_ERR_WORKSPACE;
  return KD_OK;
}

// Teacher preparation and the valid-row map: the per-call part of the loss
// that does not touch h or W.  Clears the control words first.
kd_status prepare(const int32_t* topk_idx, const float* topk_logit, const uint8_t* mask,
                  const Plan& P, float T, const Views& v, int64_t* n_valid_out, uint32_t* err,
                  cudaStream_t stream) {
  KD_CUDA(cudaMemsetAsync(v.ctrl, 0, sizeof(Ctrl), stream));
  if (P.N == 0) {
    if (n_valid_out != nullptr) KD_CUDA(cudaMemsetAsync(n_valid_out, 0, sizeof(int64_t), stream));
    return KD_OK;
  }
  KD_LAUNCH(kTeacherPrep, launch_teacher_prep(topk_idx, topk_logit, mask, P.N, static_cast<int>(P.K),
                                              P.V, T, v.row_ok, v.idx_sorted, v.p_sorted, v.plogp,
                                              v.psum, v.top1, err, stream));
  KD_LAUNCH(kCompact, launch_compact(v.row_ok, P.N, v.rows, v.ctrl, n_valid_out, stream));
  return KD_OK;
}

// The chunk loop over a prepared workspace: logsumexp pass, loss terms and,
// with want_grads, the gradient tile and both gradient products per chunk;
// then the loss.  Terms are divided by *n_norm.
kd_status chunks(const void* h, const void* W, const Plan& P, float T, float* loss,
                 float* grad_h, float* grad_W, bool want_grads, const Views& v,
                 const int64_t* n_norm, uint32_t* err, int sms, cudaStream_t stream) {
  const int64_t N = P.N, d = P.d, V = P.V;
  const kd_dtype dtype = P.dtype;
  if (N == 0) {
    KD_CUDA(cudaMemsetAsync(loss, 0, sizeof(float), stream));
    if (want_grads)
      KD_CUDA(cudaMemsetAsync(grad_W, 0, static_cast<size_t>(V) * d * sizeof(float), stream));
    return KD_OK;
  }
  const float k2 = 1.4426950408889634f / T;
  if (want_grads) KD_LAUNCH(kZeroRows, launch_zero_invalid_rows(v.row_ok, N, d, grad_h, stream));

  for (int64_t j = 0; j < P.n_chunks; ++j) {
    const NvtxRange chunk_range("chunk");
    ChunkArgs a;
    memset(&a, 0, sizeof(a));
    a.row0 = j * P.chunk;
    a.chunk = static_cast<int>(P.chunk);
    a.cpad = P.cpad;
    a.n_valid = &v.ctrl->n_valid;
    a.n_norm = n_norm;
    a.rows = v.rows;
    a.idx_sorted = v.idx_sorted;
    a.p_sorted = v.p_sorted;
    a.K = static_cast<int>(P.K);
    a.V = static_cast<int>(V);
    a.n_pb = static_cast<int>(P.n_pb);
    a.ldg = P.ldg;
    a.boff = v.boff;
    a.part_m = v.part_m;
    a.part_l = v.part_l;
    a.part_ps = v.part_ps;
    // bf16 with gradients: one reference per row, so that the gradient
    // products read the stored exponentials directly (no pass over the
    // chunk's vocabulary-wide tile between the GEMMs)
    // (the per-row values are kept for every valid row, in compacted order;
    // the kernels index them from the chunk's first row)
    const bool row_ref = dtype == KD_BF16 && want_grads;
    a.mref = row_ref ? v.mref + a.row0 : nullptr;
    a.row_flag = row_ref ? v.row_flag + a.row0 : nullptr;
    a.alpha_row = row_ref ? v.alpha_row + a.row0 : nullptr;
    a.beta_row = row_ref ? v.beta_row + a.row0 : nullptr;

    KD_LAUNCH(kGatherRows, launch_gather_rows(h, P.elem, d, a, v.hc, W, v.top1, k2, stream));
    KD_LAUNCH(kBucketOffsets, launch_bucket_offsets(a, stream));
    if (dtype == KD_BF16) {
      Pass1Args p1;
      p1.hc = v.hc;
      p1.W = W;
      p1.d = d;
      p1.k2 = k2;
      p1.row_ref = row_ref;
      // the loss alone needs no stored exponentials
      p1.u = want_grads ? static_cast<uint16_t*>(v.g) : nullptr;
      p1.counter = v.sched;
      p1.err = err;
      p1.num_sms = sms;
      KD_LAUNCH(kPass1Gemm, launch_tc_pass1(p1, a, stream));
    } else {
      KD_LAUNCH(kSimtPass1, launch_simt_pass1(static_cast<const float*>(v.hc), static_cast<const float*>(W), d,
                                a, k2, want_grads ? static_cast<float*>(v.g) : nullptr, stream));
    }
    KD_LAUNCH(kLseCombine, launch_lse(a, v.plogp, v.psum, T, v.lse, v.loss_rows, stream));
    if (!want_grads) continue;
    if (dtype == KD_BF16) {
      KD_LAUNCH(kGradPrepare, launch_grad_prepare(a, static_cast<uint16_t*>(v.g),
                                                  static_cast<uint16_t*>(v.hc), d, stream));
      KD_LAUNCH(kBwdGemm, launch_backward_gemms(v.g, W, v.hc, d, V, P.cpad, P.ldg, P.chunk, a,
                                                grad_h, grad_W, j > 0 ? 1 : 0, v.sched + 1, err,
                                                sms, stream, a.alpha_row));
    } else {
      KD_LAUNCH(kGradTile, launch_grad_tile(a, v.g, P.elem, T, stream));
      const float* G = static_cast<const float*>(v.g);
      SimtGemm gh;
      memset(&gh, 0, sizeof(gh));
      gh.A = G;
      gh.sam = P.ldg;
      gh.sak = 1;
      gh.B = static_cast<const float*>(W);
      gh.sbk = d;
      gh.sbn = 1;
      gh.C = grad_h;
      gh.ldc = d;
      gh.M_cap = P.chunk;
      gh.N = d;
      gh.Kfix = V;
      gh.m_from_count = 1;
      gh.row_map = v.rows;
      gh.row_map_off = a.row0;
      gh.n_valid = a.n_valid;
      gh.row0 = a.row0;
      KD_LAUNCH(kSimtGemm, launch_simt_gemm(gh, stream));
      SimtGemm gw;
      memset(&gw, 0, sizeof(gw));
      gw.A = G;
      gw.sam = 1;
      gw.sak = P.ldg;
      gw.B = static_cast<const float*>(v.hc);
      gw.sbk = d;
      gw.sbn = 1;
      gw.C = grad_W;
      gw.ldc = d;
      gw.M_cap = V;
      gw.N = d;
      gw.Kfix = P.chunk;
      gw.k_from_count = 1;
      gw.accumulate = j > 0 ? 1 : 0;
      gw.n_valid = a.n_valid;
      gw.row0 = a.row0;
      KD_LAUNCH(kSimtGemm, launch_simt_gemm(gw, stream));
    }
  }
  KD_LAUNCH(kFinalize, launch_finalize(v.loss_rows, v.ctrl, n_norm, loss, stream));
  return KD_OK;
}

// Pointer checks of the chunk loop's arguments.
kd_status check_outputs(const Plan& P, const void* h, const void* W, float* loss, float* grad_h,
                        float* grad_W, bool want_grads) {
  if (W == nullptr || loss == nullptr) return KD_ERR_INVALID_ARG;
  if (want_grads && grad_W == nullptr) return KD_ERR_INVALID_ARG;
  if (P.N > 0 && h == nullptr) return KD_ERR_INVALID_ARG;
  if (want_grads && P.N > 0 && grad_h == nullptr) return KD_ERR_INVALID_ARG;
  if (!aligned16(W) || (P.N > 0 && !aligned16(h))) return KD_ERR_INVALID_ARG;
  return KD_OK;
}

kd_status run(const void* h, const void* W, kd_dtype dtype, const int32_t* topk_idx,
              const float* topk_logit, const uint8_t* mask, int64_t N, int64_t d, int64_t V,
              int32_t K, float T, int64_t chunk, float* loss, float* grad_h, float* grad_W,
              bool want_grads, void* workspace, size_t ws_bytes, uint32_t* dev_err_flags,
              cudaStream_t stream) {
  const NvtxRange range(want_grads ? "kd_topk_kl_fwd_bwd" : "kd_topk_kl_fwd");
  Plan P;
  kd_status st = check_call(N, d, V, K, T, chunk, dtype, want_grads, workspace, ws_bytes, &P);
  if (st != KD_OK) return st;
  st = check_outputs(P, h, W, loss, grad_h, grad_W, want_grads);
  if (st != KD_OK) return st;
  if (N > 0 && (topk_idx == nullptr || topk_logit == nullptr)) return KD_ERR_INVALID_ARG;
  const int sms = num_sms();
  if (sms <= 0) return KD_ERR_CUDA;
  if (dtype == KD_BF16 && encode_fn() == nullptr) return KD_ERR_CUDA;
  const Views v = views(P, workspace);
  uint32_t* err = dev_err_flags != nullptr ? dev_err_flags : &v.ctrl->err;
  st = prepare(topk_idx, topk_logit, mask, P, T, v, nullptr, err, stream);
  if (st != KD_OK) return st;
  return chunks(h, W, P, T, loss, grad_h, grad_W, want_grads, v, &v.ctrl->n_valid64, err, sms,
                stream);
}

kd_status run_prepared(const void* h, const void* W, kd_dtype dtype, int64_t N, int64_t d,
                       int64_t V, int32_t K, float T, int64_t chunk, const int64_t* n_norm,
                       float* loss, float* grad_h, float* grad_W, bool want_grads,
                       void* workspace, size_t ws_bytes, uint32_t* dev_err_flags,
                       cudaStream_t stream) {
  const NvtxRange range(want_grads ? "kd_topk_kl_fwd_bwd_prepared" : "kd_topk_kl_fwd_prepared");
  Plan P;
  kd_status st = check_call(N, d, V, K, T, chunk, dtype, want_grads, workspace, ws_bytes, &P);
  if (st != KD_OK) return st;
  st = check_outputs(P, h, W, loss, grad_h, grad_W, want_grads);
  if (st != KD_OK) return st;
  const int sms = num_sms();
  if (sms <= 0) return KD_ERR_CUDA;
  if (dtype == KD_BF16 && encode_fn() == nullptr) return KD_ERR_CUDA;
  const Views v = views(P, workspace);
  uint32_t* err = dev_err_flags != nullptr ? dev_err_flags : &v.ctrl->err;
  return chunks(h, W, P, T, loss, grad_h, grad_W, want_grads, v,
                n_norm != nullptr ? n_norm : &v.ctrl->n_valid64, err, sms, stream);
}

}  // namespace
}  // namespace kd

extern "C" {

size_t kd_topk_kl_workspace_bytes(int64_t N, int64_t d, int64_t V, int32_t K, int64_t chunk,
                                  kd_dtype dtype) {
  kd::Plan p;
  if (kd::make_plan(N, d, V, K, chunk, dtype, &p) != KD_OK) return 0;
  return p.lay.total;
}

size_t kd_topk_kl_fwd_workspace_bytes(int64_t N, int64_t d, int64_t V, int32_t K, int64_t chunk,
                                      kd_dtype dtype) {
  kd::Plan p;
  if (kd::make_plan(N, d, V, K, chunk, dtype, &p) != KD_OK) return 0;
  return p.lay.off_g;
}

int64_t kd_topk_kl_default_chunk(int64_t N, int64_t d, int64_t V, kd_dtype dtype) {
  return kd::default_chunk(N, d, V, dtype);
}

kd_status kd_topk_kl_workspace_layout(int64_t N, int64_t d, int64_t V, int32_t K, int64_t chunk,
                                      kd_dtype dtype, kd_workspace_layout* out) {
  if (out == nullptr) return KD_ERR_INVALID_ARG;
  kd::Plan p;
  const kd_status st = kd::make_plan(N, d, V, K, chunk, dtype, &p);
  if (st != KD_OK) return st;
  *out = p.lay;
  return KD_OK;
}

kd_status kd_topk_kl_fwd_bwd(const void* h, const void* W, kd_dtype dtype,
                             const int32_t* topk_idx, const float* topk_logit,
                             const uint8_t* mask, int64_t N, int64_t d, int64_t V, int32_t K,
                             float T, int64_t chunk, float* loss, float* grad_h, float* grad_W,
                             void* workspace, size_t ws_bytes, uint32_t* dev_err_flags,
                             cudaStream_t stream) {
  return kd::run(h, W, dtype, topk_idx, topk_logit, mask, N, d, V, K, T, chunk, loss, grad_h,
                 grad_W, true, workspace, ws_bytes, dev_err_flags, stream);
}

kd_status kd_topk_kl_fwd(const void* h, const void* W, kd_dtype dtype, const int32_t* topk_idx,
                         const float* topk_logit, const uint8_t* mask, int64_t N, int64_t d,
                         int64_t V, int32_t K, float T, int64_t chunk, float* loss,
                         void* workspace, size_t ws_bytes, uint32_t* dev_err_flags,
                         cudaStream_t stream) {
  return kd::run(h, W, dtype, topk_idx, topk_logit, mask, N, d, V, K, T, chunk, loss, nullptr,
                 nullptr, false, workspace, ws_bytes, dev_err_flags, stream);
}

kd_status kd_topk_kl_prepare(const int32_t* topk_idx, const float* topk_logit, const uint8_t* mask,
                             int64_t N, int64_t d, int64_t V, int32_t K, float T, int64_t chunk,
                             kd_dtype dtype, void* workspace, size_t ws_bytes, int64_t* n_valid,
                             uint32_t* dev_err_flags, cudaStream_t stream) {
  const kd::NvtxRange range("kd_topk_kl_prepare");
  kd::Plan P;
  // a loss-only workspace is enough here; the chunk loop checks its own need
  kd_status st = kd::check_call(N, d, V, K, T, chunk, dtype, false, workspace, ws_bytes, &P);
  if (st != KD_OK) return st;
  if (N > 0 && (topk_idx == nullptr || topk_logit == nullptr)) return KD_ERR_INVALID_ARG;
  const kd::Views v = kd::views(P, workspace);
  uint32_t* err = dev_err_flags != nullptr ? dev_err_flags : &v.ctrl->err;
  return kd::prepare(topk_idx, topk_logit, mask, P, T, v, n_valid, err, stream);
}

kd_status kd_topk_kl_fwd_bwd_prepared(const void* h, const void* W, kd_dtype dtype, int64_t N,
                                      int64_t d, int64_t V, int32_t K, float T, int64_t chunk,
                                      const int64_t* n_norm, float* loss, float* grad_h,
                                      float* grad_W, void* workspace, size_t ws_bytes,
                                      uint32_t* dev_err_flags, cudaStream_t stream) {
  return kd::run_prepared(h, W, dtype, N, d, V, K, T, chunk, n_norm, loss, grad_h, grad_W, true,
                          workspace, ws_bytes, dev_err_flags, stream);
}

kd_status kd_topk_kl_fwd_prepared(const void* h, const void* W, kd_dtype dtype, int64_t N,
                                  int64_t d, int64_t V, int32_t K, float T, int64_t chunk,
                                  const int64_t* n_norm, float* loss, void* workspace,
                                  size_t ws_bytes, uint32_t* dev_err_flags, cudaStream_t stream) {
  return kd::run_prepared(h, W, dtype, N, d, V, K, T, chunk, n_norm, loss, nullptr, nullptr, false,
                          workspace, ws_bytes, dev_err_flags, stream);
}

kd_status kd_umma_gemm_bf16(const void* A, const void* B, float* D, int64_t M, int64_t N,
                            int64_t K, int a_mn_major, int b_mn_major, int accumulate,
                            uint32_t* counter, uint32_t* dev_err_flags, cudaStream_t stream) {
  if (A == nullptr || B == nullptr || D == nullptr || counter == nullptr ||
      dev_err_flags == nullptr)
    return KD_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1) return KD_ERR_INVALID_ARG;
  if (M >= (int64_t(1) << 30) || N >= (int64_t(1) << 30) || K >= (int64_t(1) << 30))
    return KD_ERR_UNSUPPORTED;
  const int64_t a_inner = a_mn_major ? M : K, a_outer = a_mn_major ? K : M;
  const int64_t b_inner = b_mn_major ? N : K, b_outer = b_mn_major ? K : N;
  if (a_inner % 8 != 0 || b_inner % 8 != 0) return KD_ERR_UNSUPPORTED;
  if (!kd::aligned16(A) || !kd::aligned16(B)) return KD_ERR_INVALID_ARG;
  if (kd::encode_fn() == nullptr) return KD_ERR_CUDA;
  const int sms = kd::num_sms();
  if (sms <= 0) return KD_ERR_CUDA;
  kd::TcGemmArgs g;
  memset(&g, 0, sizeof(g));
  kd::TcProblem& p = g.pr[0];
  p.A = A;
  p.a_mn = a_mn_major ? 1 : 0;
  p.a_inner = a_inner;
  p.a_outer = a_outer;
  p.lda = a_inner;
  p.B = B;
  p.b_mn = b_mn_major ? 1 : 0;
  p.b_inner = b_inner;
  p.b_outer = b_outer;
  p.ldb = b_inner;
  p.M = M;
  p.N = N;
  p.K = K;
  p.out = D;
  p.ldo = N;
  p.accumulate = accumulate ? 1 : 0;
  g.nprob = 1;
  g.chunk = static_cast<int>(M);
  g.counter = counter;
  g.err = dev_err_flags;
  g.num_sms = sms;
  return kd::launch_tc_gemm(g, stream) == cudaSuccess ? KD_OK : KD_ERR_CUDA;
}

kd_status kd_umma_gemm_bf16_wait_test(const void* A, const void* B, float* D, int64_t M,
                                      int64_t N, int64_t K, uint32_t wait_limit_us,
                                      uint32_t* counter, uint32_t* dev_err_flags,
                                      cudaStream_t stream) {
  if (A == nullptr || B == nullptr || D == nullptr || counter == nullptr ||
      dev_err_flags == nullptr || wait_limit_us == 0)
    return KD_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1) return KD_ERR_INVALID_ARG;
  if (M >= (int64_t(1) << 30) || N >= (int64_t(1) << 30) || K >= (int64_t(1) << 30) || K % 8 != 0)
    return KD_ERR_UNSUPPORTED;
  if (!kd::aligned16(A) || !kd::aligned16(B)) return KD_ERR_INVALID_ARG;
  if (kd::encode_fn() == nullptr) return KD_ERR_CUDA;
  const int sms = kd::num_sms();
  if (sms <= 0) return KD_ERR_CUDA;
  kd::TcGemmArgs g;
  memset(&g, 0, sizeof(g));
  kd::TcProblem& p = g.pr[0];
  p.A = A;
  p.a_inner = K;
  p.a_outer = M;
  p.lda = K;
  p.B = B;
  p.b_inner = K;
  p.b_outer = N;
  p.ldb = K;
  p.M = M;
  p.N = N;
  p.K = K;
  p.out = D;
  p.ldo = N;
  g.nprob = 1;
  g.chunk = static_cast<int>(M);
  g.counter = counter;
  g.err = dev_err_flags;
  g.num_sms = sms;
  g.wait_limit_ns = static_cast<uint64_t>(wait_limit_us) * 1000ull;
  g.withhold_arrival = 1;
  return kd::launch_tc_gemm(g, stream) == cudaSuccess ? KD_OK : KD_ERR_CUDA;
}

kd_status kd_timing_enable(int on) {
  std::lock_guard<std::mutex> lock(kd::g_timing_mu);
  kd::g_timing_on = on != 0;
  return KD_OK;
}

kd_status kd_timing_collect(kd_timing_entry* out, int32_t max_entries, int32_t* n_entries) {
  int64_t launches[kd::kNumKinds] = {0};
  double ms[kd::kNumKinds] = {0.0};
  kd_status st = KD_OK;
  std::vector<kd::TimingRec> recs;
  {
    std::lock_guard<std::mutex> lock(kd::g_timing_mu);
    recs.swap(kd::g_recs);
  }
  for (const kd::TimingRec& r : recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
      st = KD_ERR_CUDA;
    launches[r.kind] += 1;
    ms[r.kind] += t;
  }
  {
    std::lock_guard<std::mutex> lock(kd::g_timing_mu);
    for (const kd::TimingRec& r : recs) {
      kd::g_event_pool[r.dev].push_back(r.a);
      kd::g_event_pool[r.dev].push_back(r.b);
    }
  }
  int32_t n = 0;
  for (int k = 0; k < kd::kNumKinds; ++k) {
    if (launches[k] == 0) continue;
    if (out != nullptr && n < max_entries) {
      memset(out[n].name, 0, sizeof(out[n].name));
      strncpy(out[n].name, kd::kKindNames[k], sizeof(out[n].name) - 1);
      out[n].launches = launches[k];
      out[n].total_ms = ms[k];
    }
    ++n;
  }
  if (n_entries != nullptr) *n_entries = n;
  return st;
}

const char* kd_status_string(kd_status s) {
  switch (s) {
    case KD_OK:
      return "ok";
    case KD_ERR_INVALID_ARG:
      return "invalid argument";
    case KD_ERR_UNSUPPORTED:
      return "unsupported size";
    case KD_ERR_WORKSPACE:
      return "workspace missing or too small";
    case KD_ERR_CUDA:
      return "CUDA error";
  }
  return "unknown status";
}

}  // extern "C"
