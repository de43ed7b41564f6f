// kd_topk_cache.cu -- building the offline teacher top-K cache: the row
// kernels (per-row threshold and final selection) and the host entry point.
//
// The method keeps only the teacher's top 100 predictions per position
// ("Efficient Knowledge Distillation for LLMs: Offline Top-K Logits and a
// Fused Chunked KL Loss", ai2day.live story, "What did the researchers
// change?").  Like the loss, the cache is built without the N x V logit grid:
// per chunk of positions the tensor cores compute z = h_c W^T tile by tile
// (a leading eighth of it twice, see below), and only
// O(chunk * (V / 128 + 128 K)) numbers are kept.
//
// Every logit is compared through a 64-bit rank key (kd_tc_gemm.cu,
// rank_key): the high word orders the float, the low word makes the lower
// vocabulary index win among equal logits, so all keys of a row are distinct.
//
// A row's candidate threshold is the K-th largest of the largest keys of
// some set of its 128-column blocks: those K block maxima are K distinct keys
// at or above it, so the row's K-th largest key is too, and every top-K key
// is a candidate.  Over ALL blocks the threshold is tight: exactly K blocks
// reach it, so the candidates lie in K blocks -- at most 128 K of them
// whatever the data (ties included).  Over a sample of blocks it may be lower
// and let more candidates through, but the sample costs only its share of the
// logits.  So, per chunk of positions:
//   pass 1  the tensor cores compute the logits of the first n_s blocks only
//           (n_s = max(K, n_pb / 8), whole 256-column tiles) and keep each
//           block's largest key; tau = the K-th largest of them;
//   pass 2  all logits; each block's largest key is stored and every key
//           >= tau appended to the row's candidate list (capacity 128 K);
//   select  the K largest candidates of every row that did not overflow;
//   exact   rows that overflowed take the tight threshold from the block keys
//           of pass 2, and a third, gated pass (it returns at once when no row
//           overflowed) collects their candidates again for a second select.
// Every pass runs the same kernel with the same 256-wide tiles and the same
// accumulation order, so a logit is bit-identical in all of them.
#include <string.h>

#include <algorithm>

#include "kd_internal.h"
#include "kd_ptx.cuh"
#include "kd_topk_cache.h"

namespace kd {
namespace {

constexpr int kSelThreads = 256;

__device__ __forceinline__ float key_value(uint64_t k) {
  const uint32_t o = static_cast<uint32_t>(k >> 32);
  if (o == 0u) return __uint_as_float(0x7FC00000u);  // NaN
  const uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(u);
}

__device__ __forceinline__ int32_t key_index(uint64_t k) {
  return static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(k));
}

// The k-th largest (1-based, 1 <= k <= n) of n distinct 64-bit keys
// keys[0 .. n), by radix selection on 8-bit digits from the most significant
// one.  Per digit the first warp scans the 256-bin histogram from the top:
// lane l sums bins 255 - 8 l down to 248 - 8 l, a warp prefix sum over the
// lanes finds the lane whose bins hold the k-th key, and that lane walks its
// eight bins.  Called by every thread of the block (a multiple of 32
// threads); returns the same key to all of them.
__device__ uint64_t kth_largest(const uint64_t* __restrict__ keys, int64_t n, int64_t k) {
  __shared__ uint32_t hist[256];
  __shared__ uint64_t s_prefix;
  __shared__ int64_t s_k;
  uint64_t prefix = 0, mask = 0;
  if (threadIdx.x == 0) s_k = k;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0u;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
      const uint64_t key = keys[i];
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      uint32_t c[8];
      int64_t sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * lane - j];
        sum += c[j];
      }
      int64_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const int64_t kk = s_k;
      const int64_t excl = incl - sum;
      __syncwarp();
      if (excl < kk && kk <= incl) {
        int64_t rem = kk - excl;
        int b = 255 - 8 * lane;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (rem <= static_cast<int64_t>(c[j])) {
            b = 255 - 8 * lane - j;
            break;
          }
          rem -= c[j];
        }
        s_k = rem;
        s_prefix = prefix | (static_cast<uint64_t>(b) << shift);
      }
    }
    __syncthreads();
    prefix = s_prefix;
    mask |= static_cast<uint64_t>(255u) << shift;
  }
  return prefix;
}

// tau[i] = the K-th largest of the first nb block keys of row i (0 -- below
// every key -- when nb < K, so that every logit is a candidate).
__global__ void __launch_bounds__(kSelThreads) threshold_kernel(const uint64_t* __restrict__ bkey,
                                                                int64_t ld, int64_t nb, int64_t K,
                                                                uint64_t* __restrict__ tau) {
  const int64_t i = blockIdx.x;
  uint64_t t = 0;
  if (K <= nb) t = kth_largest(bkey + i * ld, nb, K);
  if (threadIdx.x == 0) tau[i] = t;
}

// After a pass with a sampled threshold: a row whose candidates overflowed the
// capacity gets the tight threshold over all n_pb block keys, an empty list
// and its mark set, and opens the gate of the next pass; every other row gets
// a threshold above every key, so that pass appends nothing for it.
__global__ void __launch_bounds__(kSelThreads) refine_kernel(const uint64_t* __restrict__ bkey,
                                                             int64_t n_pb, int64_t K, int64_t cap,
                                                             uint64_t* __restrict__ tau,
                                                             uint32_t* __restrict__ cnt,
                                                             uint32_t* __restrict__ redo,
                                                             uint32_t* __restrict__ gate) {
  const int64_t i = blockIdx.x;
  if (static_cast<int64_t>(cnt[i]) <= cap) {
    if (threadIdx.x == 0) {
      tau[i] = ~0ull;
      redo[i] = 0u;
    }
    return;
  }
  const uint64_t t = kth_largest(bkey + i * n_pb, n_pb, K);
  if (threadIdx.x == 0) {
    tau[i] = t;
    cnt[i] = 0u;
    redo[i] = 1u;
    atomicExch(gate, 1u);
  }
}

// The K largest candidate keys of row i, sorted, decoded into (index, logit).
//   mode 0: every row (tight thresholds: a row never overflows);
//   mode 1: rows that did not overflow (the others are redone);
//   mode 2: the redone rows only (redo[i] != 0; tight thresholds).
__global__ void __launch_bounds__(kSelThreads) select_kernel(
    const uint64_t* __restrict__ cand, int64_t cap, const uint32_t* __restrict__ cnt, int K,
    int P2, int mode, const uint32_t* __restrict__ redo, int32_t* __restrict__ out_idx,
    float* __restrict__ out_val, uint32_t* __restrict__ err) {
  extern __shared__ uint64_t skey[];
  __shared__ int s_n;
  const int64_t i = blockIdx.x;
  int64_t c = cnt[i];
  if (mode == 1 && c > cap) return;
  if (mode == 2 && redo[i] == 0u) return;
  if (c > cap) {  // cannot happen: a tight threshold bounds the candidates by 128 K
    if (threadIdx.x == 0) atomicOr(err, KD_FLAG_INTERNAL);
    c = cap;
  }
  const uint64_t* row = cand + i * cap;
  const uint64_t kth = c >= K ? kth_largest(row, c, K) : 0;
  if (threadIdx.x == 0) s_n = 0;
  for (int j = threadIdx.x; j < P2; j += blockDim.x) skey[j] = 0;
  __syncthreads();
  for (int64_t j = threadIdx.x; j < c; j += blockDim.x) {
    const uint64_t key = row[j];
    if (key >= kth) {
      const int pos = atomicAdd(&s_n, 1);
      if (pos < K) skey[pos] = key;
    }
  }
  __syncthreads();
  // bitonic sort, descending
  for (int size = 2; size <= P2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int j = threadIdx.x; j < P2; j += blockDim.x) {
        const int o = j ^ stride;
        if (o > j) {
          const bool desc = (j & size) == 0;
          const uint64_t a = skey[j], b = skey[o];
          if ((a < b) == desc) {
            skey[j] = b;
            skey[o] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  bool nan_seen = false;
  for (int j = threadIdx.x; j < K; j += blockDim.x) {
    const uint64_t key = skey[j];
    out_idx[i * K + j] = key_index(key);
    out_val[i * K + j] = key_value(key);
    nan_seen |= (key >> 32) == 0;
  }
  if (nan_seen) atomicOr(err, KD_FLAG_BAD_TEACHER);
  if (threadIdx.x == 0 && s_n != K) atomicOr(err, KD_FLAG_INTERNAL);
}

struct CachePlan {
  int64_t chunk, n_pb, cap;
  int64_t n_s;  // blocks whose logits set the first threshold
  size_t off_ctrl, off_bkey, off_tau, off_cnt, off_redo, off_cand, off_sched, total;
};

bool valid_sizes(int64_t N, int64_t d, int64_t V, int32_t K) {
  return N >= 0 && d >= 1 && V >= 1 && K >= 1 && K <= V;
}

kd_status cache_plan(int64_t N, int64_t d, int64_t V, int32_t K, int64_t chunk, CachePlan* p) {
  if (!valid_sizes(N, d, V, K)) return KD_ERR_INVALID_ARG;
  if (K > KD_MAX_K || d % 8 != 0) return KD_ERR_UNSUPPORTED;
  if (N >= (int64_t(1) << 31) || V >= (int64_t(1) << 31) - 1024 || d >= (int64_t(1) << 24))
    return KD_ERR_UNSUPPORTED;
  p->n_pb = ceil_div(V, kPB);
  p->cap = std::min<int64_t>(int64_t(kPB) * K, p->n_pb * kPB);
  // at least K blocks, an eighth of the vocabulary, whole 256-column tiles
  int64_t ns = std::max<int64_t>(K, ceil_div(p->n_pb, int64_t(8)));
  ns = round_up(ns, int64_t(kBN / kPB));
  p->n_s = std::min(ns, p->n_pb);
  int64_t c = chunk > 0 ? chunk : kd_topk_cache_default_chunk(N, V, K);
  if (N > 0 && c > N) c = N;
  if (c < 1) c = 1;
  if (c >= (int64_t(1) << 30)) return KD_ERR_UNSUPPORTED;
  p->chunk = c;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  const size_t cs = static_cast<size_t>(c);
  p->off_ctrl = take(256);
  p->off_bkey = take(8 * cs * static_cast<size_t>(p->n_pb));
  p->off_tau = take(8 * cs);
  p->off_cnt = take(4 * cs);
  p->off_redo = take(4 * cs);
  p->off_cand = take(8 * cs * static_cast<size_t>(p->cap));
  p->off_sched = take(256);
  p->total = o;
  return KD_OK;
}

}  // namespace
}  // namespace kd

extern "C" {

int64_t kd_topk_cache_default_chunk(int64_t N, int64_t V, int32_t K) {
  if (V < 1 || K < 1) return kd::kBM;
  // About 2 GiB of per-chunk buffers; equal chunks, multiples of 128 rows.
  const int64_t n_pb = kd::ceil_div(V, kd::kPB);
  const int64_t cap = std::min<int64_t>(int64_t(kd::kPB) * K, n_pb * kd::kPB);
  const int64_t per_row = 8 * (n_pb + cap + 1) + 8;
  int64_t cmax = (int64_t(2) << 30) / per_row;
  cmax = cmax / kd::kBM * kd::kBM;
  if (cmax < kd::kBM) cmax = kd::kBM;
  if (cmax > kd::kMaxChunk) cmax = kd::kMaxChunk;
  const int64_t n = N < 1 ? 1 : N;
  const int64_t pieces = kd::ceil_div(n, cmax);
  return kd::round_up(kd::ceil_div(n, pieces), kd::kBM);
}

size_t kd_topk_cache_workspace_bytes(int64_t N, int64_t d, int64_t V, int32_t K, int64_t chunk) {
  kd::CachePlan p;
  if (kd::cache_plan(N, d, V, K, chunk, &p) != KD_OK) return 0;
  return p.total;
}

kd_status kd_topk_cache_build(const void* h, const void* W, int64_t N, int64_t d, int64_t V,
                              int32_t K, int64_t chunk, int32_t* topk_idx, float* topk_logit,
                              void* workspace, size_t ws_bytes, uint32_t* dev_err_flags,
                              cudaStream_t stream) {
  const kd::NvtxRange range("kd_topk_cache_build");
  kd::CachePlan P;
  const kd_status st = kd::cache_plan(N, d, V, K, chunk, &P);
  if (st != KD_OK) return st;
  if (W == nullptr) return KD_ERR_INVALID_ARG;
  if (N > 0 && (h == nullptr || topk_idx == nullptr || topk_logit == nullptr))
    return KD_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(W) & 15u) != 0 ||
      (N > 0 && (reinterpret_cast<uintptr_t>(h) & 15u) != 0))
    return KD_ERR_INVALID_ARG;
  if (workspace == nullptr || ws_bytes < P.total) return KD_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KD_ERR_WORKSPACE;
  if (N == 0) return KD_OK;
  const int sms = kd::num_sms();
  if (sms <= 0) return KD_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* err = dev_err_flags != nullptr ? dev_err_flags : reinterpret_cast<uint32_t*>(ws + P.off_ctrl);
  uint32_t* gate = reinterpret_cast<uint32_t*>(ws + P.off_ctrl + 8);
  uint64_t* bkey = reinterpret_cast<uint64_t*>(ws + P.off_bkey);
  uint64_t* tau = reinterpret_cast<uint64_t*>(ws + P.off_tau);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(ws + P.off_cnt);
  uint32_t* redo = reinterpret_cast<uint32_t*>(ws + P.off_redo);
  uint64_t* cand = reinterpret_cast<uint64_t*>(ws + P.off_cand);
  uint32_t* sched = reinterpret_cast<uint32_t*>(ws + P.off_sched);
  if (dev_err_flags == nullptr) KD_CUDA(cudaMemsetAsync(err, 0, sizeof(uint32_t), stream));

  int P2 = 1;
  while (P2 < K) P2 <<= 1;
  const size_t sel_smem = static_cast<size_t>(P2) * sizeof(uint64_t);
  KD_CUDA(cudaFuncSetAttribute(kd::select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(sel_smem)));
  // With every block sampled the first threshold is already tight.
  const bool sampled = P.n_s < P.n_pb;
  const int64_t v_s = std::min<int64_t>(V, P.n_s * kd::kPB);

  for (int64_t row0 = 0; row0 < N; row0 += P.chunk) {
    const kd::NvtxRange chunk_range("chunk");
    const int64_t count = std::min<int64_t>(P.chunk, N - row0);
    const unsigned rows = static_cast<unsigned>(count);
    int32_t* oi = topk_idx + row0 * K;
    float* ov = topk_logit + row0 * K;
    kd::TopkGemmArgs g;
    memset(&g, 0, sizeof(g));
    g.h = static_cast<const uint8_t*>(h) + row0 * d * 2;
    g.W = W;
    g.count = count;
    g.d = d;
    g.V = V;
    g.v_cols = v_s;
    g.bkey = bkey;
    g.tau = tau;
    g.cnt = cnt;
    g.cand = cand;
    g.cap = P.cap;
    g.counter = sched;
    g.err = err;
    g.num_sms = sms;
    KD_LAUNCH(kd::kTopkBlockMax, kd::launch_tc_topk(g, 1, stream));
    KD_LAUNCH(kd::kTopkThreshold, (kd::threshold_kernel<<<rows, kd::kSelThreads, 0, stream>>>(
                                       bkey, P.n_pb, P.n_s, K, tau),
                                   cudaGetLastError()));
    KD_CUDA(cudaMemsetAsync(cnt, 0, sizeof(uint32_t) * static_cast<size_t>(count), stream));
    g.v_cols = V;
    KD_LAUNCH(kd::kTopkCandidates, kd::launch_tc_topk(g, 2, stream));
    KD_LAUNCH(kd::kTopkSelect, (kd::select_kernel<<<rows, kd::kSelThreads, sel_smem, stream>>>(
                                    cand, P.cap, cnt, K, P2, sampled ? 1 : 0, redo, oi, ov, err),
                                cudaGetLastError()));
    if (!sampled) continue;
    KD_CUDA(cudaMemsetAsync(gate, 0, sizeof(uint32_t), stream));
    KD_LAUNCH(kd::kTopkRefine, (kd::refine_kernel<<<rows, kd::kSelThreads, 0, stream>>>(
                                       bkey, P.n_pb, K, P.cap, tau, cnt, redo, gate),
                                   cudaGetLastError()));
    g.gate = gate;
    KD_LAUNCH(kd::kTopkRedo, kd::launch_tc_topk(g, 2, stream));
    KD_LAUNCH(kd::kTopkRefine, (kd::select_kernel<<<rows, kd::kSelThreads, sel_smem, stream>>>(
                                    cand, P.cap, cnt, K, P2, 2, redo, oi, ov, err),
                                cudaGetLastError()));
  }
  return KD_OK;
}

}  // extern "C"
