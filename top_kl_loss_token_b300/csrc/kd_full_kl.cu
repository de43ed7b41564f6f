// kd_full_kl.cu -- host side of the full-vocabulary (K = V) distillation
// loss: argument checks, the workspace plan and the chunk loop.
//
// Same chunked structure as kd_topk_kl_fwd_bwd ("Efficient Knowledge
// Distillation for LLMs: Offline Top-K Logits and a Fused Chunked KL Loss",
// ai2day.live story, "What did the researchers change?": chunks computed and
// discarded, no vocabulary x sequence grid), with the teacher's distribution
// computed from its hidden states and LM head in the same tensor-core pass
// instead of read from a top-K cache (the pages' online-distillation setting).
#include <math.h>
#include <string.h>

#include "kd_full_kl.h"
#include "kd_internal.h"
#include "kd_topk_kl_steps.h"

namespace kd {
namespace {

struct FullPlan {
  int64_t N, d_s, d_t, V, chunk, cpad, n_pb, ldg, n_chunks;
  size_t off_ctrl, off_row_ok, off_rows, off_lse, off_loss_rows, off_part_m, off_part_l,
      off_part_mt, off_part_lt, off_part_a, off_hc_s, off_hc_t, off_u_s, off_u_t, off_sched, total;
};

kd_status full_plan(int64_t N, int64_t d_s, int64_t d_t, int64_t V, int64_t chunk, FullPlan* p) {
  if (N < 0 || d_s < 1 || d_t < 1 || V < 1) return KD_ERR_INVALID_ARG;
  if (d_s % 8 != 0 || d_t % 8 != 0) return KD_ERR_UNSUPPORTED;
  if (N >= (int64_t(1) << 31) || V >= (int64_t(1) << 31) - 1024 || d_s >= (int64_t(1) << 24) ||
      d_t >= (int64_t(1) << 24))
    return KD_ERR_UNSUPPORTED;
  FullPlan& P = *p;
  P.N = N;
  P.d_s = d_s;
  P.d_t = d_t;
  P.V = V;
  int64_t c = chunk > 0 ? chunk : kd_full_kl_default_chunk(N, d_s, d_t, V);
  if (N > 0 && c > N) c = N;
  if (c < 1) c = 1;
  if (c >= (int64_t(1) << 30)) return KD_ERR_UNSUPPORTED;
  P.chunk = c;
  P.cpad = round_up(c, kBM);
  P.n_pb = ceil_div(V, kPB);
  P.ldg = round_up(V, kBN);
  P.n_chunks = N > 0 ? ceil_div(N, c) : 0;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  const size_t n = static_cast<size_t>(N);
  const size_t part = static_cast<size_t>(P.n_pb) * static_cast<size_t>(P.cpad);
  const size_t cp = static_cast<size_t>(P.cpad);
  P.off_ctrl = take(256);
  P.off_row_ok = take(4 * n);
  P.off_rows = take(4 * n);
  P.off_lse = take(4 * n);
  P.off_loss_rows = take(4 * n);
  P.off_part_m = take(4 * part);
  P.off_part_l = take(4 * part);
  P.off_part_mt = take(4 * part);
  P.off_part_lt = take(4 * part);
  P.off_part_a = take(4 * part);
  P.off_hc_s = take(cp * static_cast<size_t>(d_s) * 2);
  P.off_hc_t = take(cp * static_cast<size_t>(d_t) * 2);
  P.off_u_s = take(cp * static_cast<size_t>(P.ldg) * 2);
  P.off_u_t = take(cp * static_cast<size_t>(P.ldg) * 2);
  P.off_sched = take(256);
  P.total = o;
  return KD_OK;
}

}  // namespace
}  // namespace kd

extern "C" {

int64_t kd_full_kl_default_chunk(int64_t N, int64_t d_s, int64_t d_t, int64_t V) {
  // Both models' exponential tiles (2 x chunk x V bf16) near 8 GiB; both
  // models' hidden states of the chunk resident in L2 (at 32K tokens,
  // d_s = d_t = 2880, V = 201,088, on one GPU: chunk 8192 133.5 ms per step,
  // 5504 130.7, 4096 127.3; on another: 4096 125.4, 3072 126.3, 2048 129.5);
  // equal chunks, multiples of 128 rows.
  const int64_t ldg = kd::round_up(V < 1 ? 1 : V, kd::kBN);
  int64_t cmax = (int64_t(8) << 30) / (4 * ldg);
  cmax = cmax / kd::kBM * kd::kBM;
  if (cmax < kd::kBM) cmax = kd::kBM;
  if (cmax > kd::kMaxChunk) cmax = kd::kMaxChunk;
  const int64_t cl2 = kd::l2_chunk_cap(2 * ((d_s < 1 ? 1 : d_s) + (d_t < 1 ? 1 : d_t)));
  if (cmax > cl2) cmax = cl2;
  const int64_t n = N < 1 ? 1 : N;
  const int64_t pieces = kd::ceil_div(n, cmax);
  return kd::round_up(kd::ceil_div(n, pieces), kd::kBM);
}

size_t kd_full_kl_workspace_bytes(int64_t N, int64_t d_s, int64_t d_t, int64_t V, int64_t chunk) {
  kd::FullPlan p;
  if (kd::full_plan(N, d_s, d_t, V, chunk, &p) != KD_OK) return 0;
  return p.total;
}

kd_status kd_full_kl_workspace_layout(int64_t N, int64_t d_s, int64_t d_t, int64_t V,
                                      int64_t chunk, kd_workspace_layout* out) {
  if (out == nullptr) return KD_ERR_INVALID_ARG;
  kd::FullPlan p;
  const kd_status st = kd::full_plan(N, d_s, d_t, V, chunk, &p);
  if (st != KD_OK) return st;
  memset(out, 0, sizeof(*out));
  out->chunk = p.chunk;
  out->chunk_pad = p.cpad;
  out->n_pb = p.n_pb;
  out->ld_g = p.ldg;
  out->off_ctrl = p.off_ctrl;
  out->off_row_ok = p.off_row_ok;
  out->off_rows = p.off_rows;
  out->off_lse = p.off_lse;
  out->off_loss_rows = p.off_loss_rows;
  out->off_part_m = p.off_part_m;
  out->off_part_l = p.off_part_l;
  out->off_hc = p.off_hc_s;
  out->off_g = p.off_u_s;
  out->off_sched = p.off_sched;
  out->total = p.total;
  return KD_OK;
}

kd_status kd_full_kl_fwd_bwd(const void* h_s, const void* W_s, const void* h_t, const void* W_t,
                             const uint8_t* mask, int64_t N, int64_t d_s, int64_t d_t, int64_t V,
                             float T, int64_t chunk, float* loss, float* grad_h, float* grad_W,
                             void* workspace, size_t ws_bytes, uint32_t* dev_err_flags,
                             cudaStream_t stream) {
  const kd::NvtxRange range("kd_full_kl_fwd_bwd");
  kd::FullPlan P;
  const kd_status st = kd::full_plan(N, d_s, d_t, V, chunk, &P);
  if (st != KD_OK) return st;
  if (!(T > 0.f) || !isfinite(T)) return KD_ERR_INVALID_ARG;
  if (W_s == nullptr || W_t == nullptr || loss == nullptr || grad_W == nullptr)
    return KD_ERR_INVALID_ARG;
  if (N > 0 && (h_s == nullptr || h_t == nullptr || grad_h == nullptr)) return KD_ERR_INVALID_ARG;
  if (!kd::aligned16(W_s) || !kd::aligned16(W_t) ||
      (N > 0 && (!kd::aligned16(h_s) || !kd::aligned16(h_t))))
    return KD_ERR_INVALID_ARG;
  if (workspace == nullptr || ws_bytes < P.total) return KD_ERR_WORKSPACE;
  if (!kd::aligned16(workspace)) return KD_ERR_WORKSPACE;
  const int sms = kd::num_sms();
  if (sms <= 0) return KD_ERR_CUDA;

  uint8_t* b = static_cast<uint8_t*>(workspace);
  kd::Ctrl* ctrl = reinterpret_cast<kd::Ctrl*>(b + P.off_ctrl);
  int32_t* row_ok = reinterpret_cast<int32_t*>(b + P.off_row_ok);
  int32_t* rows = reinterpret_cast<int32_t*>(b + P.off_rows);
  float* lse = reinterpret_cast<float*>(b + P.off_lse);
  float* loss_rows = reinterpret_cast<float*>(b + P.off_loss_rows);
  float* part_m = reinterpret_cast<float*>(b + P.off_part_m);
  float* part_l = reinterpret_cast<float*>(b + P.off_part_l);
  float* part_mt = reinterpret_cast<float*>(b + P.off_part_mt);
  float* part_lt = reinterpret_cast<float*>(b + P.off_part_lt);
  float* part_a = reinterpret_cast<float*>(b + P.off_part_a);
  void* hc_s = b + P.off_hc_s;
  void* hc_t = b + P.off_hc_t;
  uint16_t* u_s = reinterpret_cast<uint16_t*>(b + P.off_u_s);
  uint16_t* u_t = reinterpret_cast<uint16_t*>(b + P.off_u_t);
  uint32_t* sched = reinterpret_cast<uint32_t*>(b + P.off_sched);
  uint32_t* err = dev_err_flags != nullptr ? dev_err_flags : &ctrl->err;

  KD_CUDA(cudaMemsetAsync(ctrl, 0, sizeof(kd::Ctrl), stream));
  if (N == 0) {
    KD_CUDA(cudaMemsetAsync(loss, 0, sizeof(float), stream));
    KD_CUDA(cudaMemsetAsync(grad_W, 0, static_cast<size_t>(V) * d_s * sizeof(float), stream));
    return KD_OK;
  }
  KD_LAUNCH(kd::kMaskRows, kd::launch_mask_rows(mask, N, row_ok, stream));
  KD_LAUNCH(kd::kCompact, kd::launch_compact(row_ok, N, rows, ctrl, nullptr, stream));
  KD_LAUNCH(kd::kZeroRows, kd::launch_zero_invalid_rows(row_ok, N, d_s, grad_h, stream));

  for (int64_t j = 0; j < P.n_chunks; ++j) {
    const kd::NvtxRange chunk_range("chunk");
    kd::ChunkArgs a;
    memset(&a, 0, sizeof(a));
    a.row0 = j * P.chunk;
    a.chunk = static_cast<int>(P.chunk);
    a.cpad = P.cpad;
    a.n_valid = &ctrl->n_valid;
    a.n_norm = &ctrl->n_valid64;
    a.rows = rows;
    a.V = static_cast<int>(V);
    a.n_pb = static_cast<int>(P.n_pb);
    a.ldg = P.ldg;
    a.part_m = part_m;
    a.part_l = part_l;

    KD_LAUNCH(kd::kGatherRows,
              kd::launch_gather_rows(h_s, 2, d_s, a, hc_s, nullptr, nullptr, 0.f, stream));
    KD_LAUNCH(kd::kGatherRows,
              kd::launch_gather_rows(h_t, 2, d_t, a, hc_t, nullptr, nullptr, 0.f, stream));
    kd::DualPass1Args p1;
    memset(&p1, 0, sizeof(p1));
    p1.hc_t = hc_t;
    p1.W_t = W_t;
    p1.hc_s = hc_s;
    p1.W_s = W_s;
    p1.d_t = d_t;
    p1.d_s = d_s;
    p1.k2 = 1.4426950408889634f / T;
    p1.u_t = u_t;
    p1.u_s = u_s;
    p1.part_mt = part_mt;
    p1.part_lt = part_lt;
    p1.part_a = part_a;
    p1.counter = sched;
    p1.err = err;
    p1.num_sms = sms;
    KD_LAUNCH(kd::kFullPass1Gemm, kd::launch_tc_dual_pass1(p1, a, stream));
    KD_LAUNCH(kd::kFullLseCombine,
              kd::launch_lse_dual(a, part_mt, part_lt, part_a, T, lse, loss_rows, stream));
    KD_LAUNCH(kd::kFullGradTile, kd::launch_grad_tile_dual(a, part_mt, u_t, u_s, stream));
    KD_LAUNCH(kd::kBwdGemm, kd::launch_backward_gemms(u_s, W_s, hc_s, d_s, V, P.cpad, P.ldg,
                                                      P.chunk, a, grad_h, grad_W, j > 0 ? 1 : 0,
                                                      sched + 1, err, sms, stream));
  }
  KD_LAUNCH(kd::kFinalize, kd::launch_finalize(loss_rows, ctrl, &ctrl->n_valid64, loss, stream));
  return KD_OK;
}

}  // extern "C"
