// kd_rowops.cu -- the row-wise kernels of the fused top-K KL loss and its
// fp32 CUDA-core path.
//
// "Efficient Knowledge Distillation for LLMs: Offline Top-K Logits and a Fused
// Chunked KL Loss" keeps only the teacher's top K (index, logit) pairs per
// position (ai2day.live story, "What did the researchers change?") and drops
// the rest of the teacher distribution (elseif.net summary, third paragraph).
// These kernels turn that cache into renormalised probabilities, combine the
// per-block logsumexp statistics of the student logits into the per-token
// loss, form the gradient of the loss with respect to the logits one chunk at
// a time, and reduce the loss.  Every exponential is taken in base 2:
// s2 = z * log2(e) / T, so softmax(z / T) = 2^(s2 - lse2).
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include "kd_internal.h"
#include "kd_ptx.cuh"

namespace kd {
namespace {

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ int chunk_count(const int32_t* n_valid, int64_t row0, int chunk) {
  const long long c = static_cast<long long>(*n_valid) - row0;
  return c < 0 ? 0 : (c > chunk ? chunk : static_cast<int>(c));
}

// 1 / (T n) for the loss's divisor n; 0 when n <= 0 (no valid token anywhere).
__device__ __forceinline__ float grad_scale(const int64_t* n_norm, float T) {
  const int64_t n = *n_norm;
  return n > 0 ? 1.0f / (T * static_cast<float>(n)) : 0.f;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_or(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------------------- teacher prep
//
// One block per token row r:
//   valid row     mask[r] != 0 (or no mask) and a usable teacher row;
//   drop          entries whose index is outside [0, V) (flag INDEX_RANGE);
//   bad row       a NaN or +inf among the in-range logits, or no finite one
//                 (flag BAD_TEACHER; the row is then treated as masked);
//   p_k           = 2^(t2_k - max t2) / sum, t2 = logit * log2(e) / T
//                 (renormalised over the kept entries, -inf -> 0);
//   plogp         = sum_k p_k ln p_k,  psum = sum_k p_k;
//   sorted list   the kept (index, p) pairs in increasing index order,
//                 padded with (kNoIndex, 0) up to K.
constexpr int kPrepThreads = 128;

__global__ void __launch_bounds__(kPrepThreads) teacher_prep_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ logit,
    const uint8_t* __restrict__ mask, int K, int64_t V, float k2, int P2,
    int32_t* __restrict__ row_ok, int32_t* __restrict__ idx_sorted,
    float* __restrict__ p_sorted, float* __restrict__ plogp, float* __restrict__ psum,
    int32_t* __restrict__ top1, uint32_t* __restrict__ err) {
  extern __shared__ uint8_t sm[];
  int32_t* skey = reinterpret_cast<int32_t*>(sm);
  float* sval = reinterpret_cast<float*>(skey + P2);
  __shared__ float red_f[kPrepThreads / 32];
  __shared__ int red_i[kPrepThreads / 32];

  const int64_t r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (mask != nullptr && mask[r] == 0) {
    if (tid == 0) row_ok[r] = 0;
    return;
  }
  const int32_t* ri = idx + r * K;
  const float* rl = logit + r * K;

  // Pass A: drop out-of-range entries, find bad rows, max of t2.
  int bits = 0;  // 1: out of range seen, 2: NaN / +inf seen, 4: finite seen
  float mx = -INFINITY;
  for (int k = tid; k < P2; k += kPrepThreads) {
    int key = kNoIndex;
    float t2 = -INFINITY;
    if (k < K) {
      const int32_t v = ri[k];
      const float l = rl[k];
      if (v < 0 || static_cast<int64_t>(v) >= V) {
        bits |= 1;
      } else {
        key = v;
        if (isnan(l) || l == INFINITY) bits |= 2;
        if (isfinite(l)) bits |= 4;
        t2 = l * k2;
        mx = fmaxf(mx, t2);
      }
    }
    skey[k] = key;
    sval[k] = t2;
  }
  bits = warp_or(bits);
  mx = warp_max(mx);
  if (lane == 0) {
    red_i[wid] = bits;
    red_f[wid] = mx;
  }
  __syncthreads();
  bits = 0;
  mx = -INFINITY;
#pragma unroll
  for (int w = 0; w < kPrepThreads / 32; ++w) {
    bits |= red_i[w];
    mx = fmaxf(mx, red_f[w]);
  }
  __syncthreads();
  const bool bad = (bits & 2) || !(bits & 4);
  if (tid == 0) {
    uint32_t f = 0;
    if (bits & 1) f |= KD_FLAG_INDEX_RANGE;
    if (bad) f |= KD_FLAG_BAD_TEACHER;
    if (f) atomicOr(err, f);
    row_ok[r] = bad ? 0 : 1;
  }
  if (bad) return;

  // Pass B: exponentials and their sum.
  float sum = 0.f;
  for (int k = tid; k < P2; k += kPrepThreads) {
    const float e = (skey[k] != kNoIndex) ? ex2_approx(sval[k] - mx) : 0.f;
    sval[k] = e;
    sum += e;
  }
  sum = warp_sum(sum);
  if (lane == 0) red_f[wid] = sum;
  __syncthreads();
  sum = 0.f;
#pragma unroll
  for (int w = 0; w < kPrepThreads / 32; ++w) sum += red_f[w];
  __syncthreads();

  // Pass C: probabilities, sum p ln p, sum p, and the most probable entry
  // (the lower index among equal probabilities).
  const float inv = 1.0f / sum;
  const float lgsum = lg2_approx(sum);
  float pl = 0.f, ps = 0.f;
  float pbest = -1.f;
  int ibest = kNoIndex;
  for (int k = tid; k < P2; k += kPrepThreads) {
    const float e = sval[k];
    const float p = e * inv;
    if (p > 0.f) {
      // ln p = ln(e) - ln(sum) with ln(e) = log2(e) * ln 2
      pl += p * (lg2_approx(e) - lgsum) * kLn2;
    }
    if (skey[k] != kNoIndex && (p > pbest || (p == pbest && skey[k] < ibest))) {
      pbest = p;
      ibest = skey[k];
    }
    ps += p;
    sval[k] = p;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float po = __shfl_xor_sync(0xffffffffu, pbest, o);
    const int io = __shfl_xor_sync(0xffffffffu, ibest, o);
    if (po > pbest || (po == pbest && io < ibest)) {
      pbest = po;
      ibest = io;
    }
  }
  __shared__ float red_pb[kPrepThreads / 32];
  __shared__ int red_ib[kPrepThreads / 32];
  pl = warp_sum(pl);
  ps = warp_sum(ps);
  if (lane == 0) {
    red_f[wid] = pl;
    red_i[wid] = __float_as_int(ps);
    red_pb[wid] = pbest;
    red_ib[wid] = ibest;
  }
  __syncthreads();
  if (tid == 0) {
    float a = 0.f, b = 0.f;
    float pb = -1.f;
    int ib = kNoIndex;
#pragma unroll
    for (int w = 0; w < kPrepThreads / 32; ++w) {
      a += red_f[w];
      b += __int_as_float(red_i[w]);
      if (red_pb[w] > pb || (red_pb[w] == pb && red_ib[w] < ib)) {
        pb = red_pb[w];
        ib = red_ib[w];
      }
    }
    plogp[r] = a;
    psum[r] = b;
    if (top1 != nullptr) top1[r] = ib;
  }

  // Bitonic sort of (key, p) by key over P2 (a power of two) slots.
  for (int size = 2; size <= P2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int k = tid; k < P2; k += kPrepThreads) {
        const int o = k ^ stride;
        if (o > k) {
          const bool up = (k & size) == 0;
          const int a = skey[k], b = skey[o];
          if ((a > b) == up) {
            skey[k] = b;
            skey[o] = a;
            const float t = sval[k];
            sval[k] = sval[o];
            sval[o] = t;
          }
        }
      }
    }
  }
  __syncthreads();
  for (int k = tid; k < K; k += kPrepThreads) {
    idx_sorted[r * K + k] = skey[k];
    p_sorted[r * K + k] = (skey[k] == kNoIndex) ? 0.f : sval[k];
  }
}

// The same teacher preparation with one warp per row, for K <= 128: each lane
// keeps E = P2 / 32 entries in registers (entry g = lane + 32 e), the
// reductions are warp shuffles and the sort is a bitonic network across lanes
// (shuffles) and registers (swaps), so no block-wide barrier is needed.  Four
// rows per block.
constexpr int kPrepWarpRows = 4;

template <int E>
__global__ void __launch_bounds__(32 * kPrepWarpRows) teacher_prep_warp_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ logit,
    const uint8_t* __restrict__ mask, int64_t N, int K, int64_t V, float k2,
    int32_t* __restrict__ row_ok, int32_t* __restrict__ idx_sorted,
    float* __restrict__ p_sorted, float* __restrict__ plogp, float* __restrict__ psum,
    int32_t* __restrict__ top1, uint32_t* __restrict__ err) {
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * kPrepWarpRows + (threadIdx.x >> 5);
  if (r >= N) return;
  if (mask != nullptr && mask[r] == 0) {
    if (lane == 0) row_ok[r] = 0;
    return;
  }
  const int32_t* ri = idx + r * K;
  const float* rl = logit + r * K;
  int key[E];
  float val[E];
  int bits = 0;  // 1: out of range seen, 2: NaN / +inf seen, 4: finite seen
  float mx = -INFINITY;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int k = lane + 32 * e;
    key[e] = kNoIndex;
    val[e] = -INFINITY;
    if (k < K) {
      const int32_t v = ri[k];
      const float l = rl[k];
      if (v < 0 || static_cast<int64_t>(v) >= V) {
        bits |= 1;
      } else {
        key[e] = v;
        if (isnan(l) || l == INFINITY) bits |= 2;
        if (isfinite(l)) bits |= 4;
        val[e] = l * k2;
        mx = fmaxf(mx, val[e]);
      }
    }
  }
  bits = warp_or(bits);
  mx = warp_max(mx);
  const bool bad = (bits & 2) || !(bits & 4);
  if (lane == 0) {
    uint32_t f = 0;
    if (bits & 1) f |= KD_FLAG_INDEX_RANGE;
    if (bad) f |= KD_FLAG_BAD_TEACHER;
    if (f) atomicOr(err, f);
    row_ok[r] = bad ? 0 : 1;
  }
  if (bad) return;
  float sum = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    val[e] = (key[e] != kNoIndex) ? ex2_approx(val[e] - mx) : 0.f;
    sum += val[e];
  }
  sum = warp_sum(sum);
  const float inv = 1.0f / sum;
  const float lgsum = lg2_approx(sum);
  float pl = 0.f, ps = 0.f, pbest = -1.f;
  int ibest = kNoIndex;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const float ex = val[e];
    const float p = ex * inv;
    if (p > 0.f) pl += p * (lg2_approx(ex) - lgsum) * kLn2;
    if (key[e] != kNoIndex && (p > pbest || (p == pbest && key[e] < ibest))) {
      pbest = p;
      ibest = key[e];
    }
    ps += p;
    val[e] = p;
  }
  pl = warp_sum(pl);
  ps = warp_sum(ps);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float po = __shfl_xor_sync(0xffffffffu, pbest, o);
    const int io = __shfl_xor_sync(0xffffffffu, ibest, o);
    if (po > pbest || (po == pbest && io < ibest)) {
      pbest = po;
      ibest = io;
    }
  }
  if (lane == 0) {
    plogp[r] = pl;
    psum[r] = ps;
    if (top1 != nullptr) top1[r] = ibest;
  }
  // Bitonic sort of (key, p) by key over P2 = 32 E slots, slot g = lane + 32 e.
#pragma unroll
  for (int size = 2; size <= 32 * E; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int g = lane + 32 * e;
        const int og = g ^ stride;
        if (stride < 32) {
          const int ok = __shfl_xor_sync(0xffffffffu, key[e], stride);
          const float ov = __shfl_xor_sync(0xffffffffu, val[e], stride);
          const bool up = (g & size) == 0;
          // the lower slot of the pair keeps the smaller key when ascending
          const bool keep_small = (g < og) == up;
          const bool take = keep_small ? (ok < key[e]) : (ok > key[e]);
          if (take) {
            key[e] = ok;
            val[e] = ov;
          }
        } else if (og > g) {
          const int eo = e ^ (stride >> 5);
          const bool up = (g & size) == 0;
          if ((key[e] > key[eo]) == up) {
            const int tk = key[e];
            key[e] = key[eo];
            key[eo] = tk;
            const float tv = val[e];
            val[e] = val[eo];
            val[eo] = tv;
          }
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int k = lane + 32 * e;
    if (k < K) {
      idx_sorted[r * K + k] = key[e];
      p_sorted[r * K + k] = (key[e] == kNoIndex) ? 0.f : val[e];
    }
  }
}

// ------------------------------------------------------------- compaction
// One block: rows[i] = the i-th row with row_ok != 0, n_valid = their count.
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads) compact_kernel(const int32_t* __restrict__ row_ok,
                                                              int64_t N,
                                                              int32_t* __restrict__ rows,
                                                              Ctrl* ctrl,
                                                              int64_t* __restrict__ n_valid_out) {
  __shared__ int warp_tot[kScanThreads / 32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int64_t base = 0; base < N; base += kScanThreads) {
    const int64_t r = base + tid;
    const int f = (r < N && row_ok[r] != 0) ? 1 : 0;
    const uint32_t bal = __ballot_sync(0xffffffffu, f);
    const int before = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) warp_tot[wid] = __popc(bal);
    __syncthreads();
    int off = 0, tot = 0;
    for (int w = 0; w < kScanThreads / 32; ++w) {
      const int c = warp_tot[w];
      if (w < wid) off += c;
      tot += c;
    }
    if (f) rows[carry + off + before] = static_cast<int32_t>(r);
    __syncthreads();
    if (tid == 0) carry += tot;
    __syncthreads();
  }
  if (tid == 0) {
    ctrl->n_valid = carry;
    ctrl->n_valid64 = carry;
    ctrl->loss_sum = 0.0;
    if (n_valid_out != nullptr) *n_valid_out = carry;
  }
}

// ------------------------------------------------------------- per-chunk kernels

// hc[i, :] = h[rows[row0 + i], :] for the chunk's valid rows; zero rows up to
// the next multiple of 128 so the tensor-core tiles never read stale data.
// With a.mref (bf16 only): also row i's reference m_i = k2 * (h_r . W[top1_r]),
// the student's logit at the teacher's most probable entry in log2 units (a
// value the row's logits reach, so exponentials relative to it stay in
// range), and a cleared row flag.
constexpr int kGatherThreads = 128;

__global__ void __launch_bounds__(kGatherThreads) gather_rows_kernel(
    const uint8_t* __restrict__ h, int64_t row_bytes, ChunkArgs a, uint8_t* __restrict__ hc,
    const uint8_t* __restrict__ W, const int32_t* __restrict__ top1, float k2) {
  const int i = blockIdx.x;
  const int count = chunk_count(a.n_valid, a.row0, a.chunk);
  if (i >= round_up(count, 128)) return;
  uint4* dst = reinterpret_cast<uint4*>(hc + static_cast<int64_t>(i) * row_bytes);
  const int64_t n16 = row_bytes / 16;
  if (i < count) {
    const int64_t r = a.rows[a.row0 + i];
    const uint4* src = reinterpret_cast<const uint4*>(h + r * row_bytes);
    if (a.mref == nullptr) {
      for (int64_t j = threadIdx.x; j < n16; j += blockDim.x) dst[j] = src[j];
      return;
    }
    const uint4* wrow = reinterpret_cast<const uint4*>(W + static_cast<int64_t>(top1[r]) * row_bytes);
    float dot = 0.f;
    for (int64_t j = threadIdx.x; j < n16; j += blockDim.x) {
      const uint4 x = src[j];
      const uint4 w = __ldg(wrow + j);
      dst[j] = x;
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        dot = fmaf(bf16lo_to_f32(xs[q]), bf16lo_to_f32(ws[q]), dot);
        dot = fmaf(bf16hi_to_f32(xs[q]), bf16hi_to_f32(ws[q]), dot);
      }
    }
    __shared__ float red[kGatherThreads / 32];
    dot = warp_sum(dot);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = dot;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < kGatherThreads / 32; ++w) t += red[w];
      a.mref[i] = t * k2;
      a.row_flag[i] = 0;
    }
  } else {
    for (int64_t j = threadIdx.x; j < n16; j += blockDim.x) dst[j] = make_uint4(0, 0, 0, 0);
    if (a.mref != nullptr && threadIdx.x == 0) {
      a.mref[i] = 0.f;
      a.row_flag[i] = 0;
    }
  }
}

// boff[pb][i] = first position in row i's sorted list whose index is >= pb*128,
// for pb = 0 .. n_pb (the last one is the number of kept entries).
constexpr int kBoffRows = 64;
constexpr int kBoffGroups = 4;
constexpr int kBoffPerThread = 64;

__global__ void __launch_bounds__(kBoffRows * kBoffGroups) bucket_offsets_kernel(ChunkArgs a) {
  const int count = chunk_count(a.n_valid, a.row0, a.chunk);
  const int i = blockIdx.x * kBoffRows + threadIdx.x;
  if (i >= count) return;
  const int pb0 = (blockIdx.y * kBoffGroups + threadIdx.y) * kBoffPerThread;
  if (pb0 > a.n_pb) return;
  const int pb1 = min(pb0 + kBoffPerThread, a.n_pb + 1);
  const int32_t* lst = a.idx_sorted + static_cast<int64_t>(a.rows[a.row0 + i]) * a.K;
  // lower bound of pb0 * 128
  const int target0 = pb0 * kPB;
  int lo = 0, hi = a.K;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(lst + mid) < target0) lo = mid + 1;
    else hi = mid;
  }
  // the next entry's index stays in a register: most blocks hold no entry,
  // so the loop is a compare and a store per block
  int off = lo;
  int nxt = off < a.K ? __ldg(lst + off) : INT_MAX;
  for (int pb = pb0; pb < pb1; ++pb) {
    const int target = pb * kPB;
    while (nxt < target) {
      ++off;
      nxt = off < a.K ? __ldg(lst + off) : INT_MAX;
    }
    a.boff[static_cast<int64_t>(pb) * a.cpad + i] = static_cast<uint16_t>(off);
  }
}

// Combine the per-block statistics of each row of the chunk:
//   lse2 = M + log2(sum_b l_b 2^(m_b - M)),  M = max_b m_b
//   loss_i = plogp - ln2 * (sum_b ps_b - psum * lse2)
// then overwrite part_m with alpha_b = 2^(m_b - lse2) / (T N_valid), the factor
// that turns the stored exponentials of block b into softmax / (T N_valid).
constexpr int kLseRows = 32;
constexpr int kLseGroups = 16;

__global__ void __launch_bounds__(kLseRows * kLseGroups) lse_kernel(
    ChunkArgs a, const float* __restrict__ plogp, const float* __restrict__ psum, float T,
    float* __restrict__ lse_out, float* __restrict__ loss_rows) {
  __shared__ float sM[kLseGroups][kLseRows];
  __shared__ float sL[kLseGroups][kLseRows];
  __shared__ float sP[kLseGroups][kLseRows];
  __shared__ float sLse[kLseRows];
  const int count = chunk_count(a.n_valid, a.row0, a.chunk);
  const int i0 = blockIdx.x * kLseRows;
  if (i0 >= count) return;
  const int x = threadIdx.x, y = threadIdx.y;
  const int i = i0 + x;
  const bool live = i < count;
  float M = -INFINITY, L = 0.f, PS = 0.f;
  if (live) {
    // four blocks' statistics loaded before they are combined, so that
    // several loads per thread are in flight
    int pb = y;
    for (; pb + 3 * kLseGroups < a.n_pb; pb += 4 * kLseGroups) {
      float m[4], l[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t o = static_cast<int64_t>(pb + u * kLseGroups) * a.cpad + i;
        m[u] = a.part_m[o];
        l[u] = a.part_l[o];
        PS += a.part_ps[o];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (m[u] > M) {
          L = L * ex2_approx(M - m[u]) + l[u];
          M = m[u];
        } else {
          L += l[u] * ex2_approx(m[u] - M);
        }
      }
    }
    for (; pb < a.n_pb; pb += kLseGroups) {
      const int64_t o = static_cast<int64_t>(pb) * a.cpad + i;
      const float m = a.part_m[o], l = a.part_l[o];
      PS += a.part_ps[o];
      if (m > M) {
        L = L * ex2_approx(M - m) + l;
        M = m;
      } else {
        L += l * ex2_approx(m - M);
      }
    }
  }
  sM[y][x] = M;
  sL[y][x] = L;
  sP[y][x] = PS;
  __syncthreads();
  if (y == 0 && live) {
    float MM = -INFINITY;
    for (int g = 0; g < kLseGroups; ++g) MM = fmaxf(MM, sM[g][x]);
    float LL = 0.f, PP = 0.f;
    for (int g = 0; g < kLseGroups; ++g) {
      LL += sL[g][x] * ex2_approx(sM[g][x] - MM);
      PP += sP[g][x];
    }
    const float lse2 = MM + lg2_approx(LL);
    const int64_t r = a.rows[a.row0 + i];
    const float loss = plogp[r] - kLn2 * (PP - psum[r] * lse2);
    lse_out[a.row0 + i] = lse2 * kLn2;
    loss_rows[a.row0 + i] = loss;
    sLse[x] = lse2;
    if (a.alpha_row != nullptr) {
      // MM is the row's common reference: its own m_i, or, when some block
      // kept its own maximum, the largest block reference (the row is then
      // rescaled to it before the gradient products); it replaces m_i
      a.alpha_row[i] = ex2_approx(MM - lse2) * grad_scale(a.n_norm, T);
      a.beta_row[i] = ex2_approx(lse2 - MM);
      a.mref[i] = MM;
    }
  }
  // One reference per row: the gradient products need no per-block factor
  // (grad_prepare rescales the rare rows with several references from the
  // block references themselves).
  if (a.alpha_row != nullptr) return;
  __syncthreads();
  if (!live) return;
  const float lse2 = sLse[x];
  const float scale = grad_scale(a.n_norm, T);
  for (int pb = y; pb < a.n_pb; pb += kLseGroups) {
    const int64_t o = static_cast<int64_t>(pb) * a.cpad + i;
    a.part_m[o] = ex2_approx(a.part_m[o] - lse2) * scale;
  }
}

// G[i, v] = u[i, v] * alpha_{block(v)} - (sum of p over teacher entries at v) / (T N_valid),
// written in place over u.  Rows count .. round_up(count, 64) are zeroed (the
// grad_W reduction reads whole 64-row blocks); columns >= V are zeroed.
template <typename E>
struct GVec;
template <>
struct GVec<uint16_t> {
  static constexpr int kW = 8;
  __device__ static void load(const uint16_t* p, float (&f)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    f[0] = bf16lo_to_f32(v.x);
    f[1] = bf16hi_to_f32(v.x);
    f[2] = bf16lo_to_f32(v.y);
    f[3] = bf16hi_to_f32(v.y);
    f[4] = bf16lo_to_f32(v.z);
    f[5] = bf16hi_to_f32(v.z);
    f[6] = bf16lo_to_f32(v.w);
    f[7] = bf16hi_to_f32(v.w);
  }
  __device__ static void store(uint16_t* p, const float (&f)[8]) {
    *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                              pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
  }
};
template <>
struct GVec<float> {
  static constexpr int kW = 4;
  __device__ static void load(const float* p, float (&f)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    f[0] = v.x;
    f[1] = v.y;
    f[2] = v.z;
    f[3] = v.w;
  }
  __device__ static void store(float* p, const float (&f)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
  }
};

constexpr int kGThreads = 256;

template <typename E>
__global__ void __launch_bounds__(kGThreads) grad_tile_kernel(ChunkArgs a, E* __restrict__ g,
                                                              float T) {
  constexpr int W = GVec<E>::kW;
  extern __shared__ uint8_t sm[];
  float* salpha = reinterpret_cast<float*>(sm);
  uint16_t* sboff = reinterpret_cast<uint16_t*>(salpha + a.n_pb);
  const int count = chunk_count(a.n_valid, a.row0, a.chunk);
  const int i = blockIdx.x;
  if (i >= round_up(count, 64)) return;
  E* row = g + static_cast<int64_t>(i) * a.ldg;
  if (i >= count) {
    float z[W];
#pragma unroll
    for (int j = 0; j < W; ++j) z[j] = 0.f;
    for (int64_t v0 = static_cast<int64_t>(threadIdx.x) * W; v0 < a.ldg; v0 += kGThreads * W)
      GVec<E>::store(row + v0, z);
    return;
  }
  for (int pb = threadIdx.x; pb < a.n_pb; pb += kGThreads) {
    salpha[pb] = a.part_m[static_cast<int64_t>(pb) * a.cpad + i];
    sboff[pb] = a.boff[static_cast<int64_t>(pb) * a.cpad + i];
  }
  if (threadIdx.x == 0) sboff[a.n_pb] = a.boff[static_cast<int64_t>(a.n_pb) * a.cpad + i];
  __syncthreads();
  const int64_t r = a.rows[a.row0 + i];
  const int32_t* lidx = a.idx_sorted + r * a.K;
  const float* lp = a.p_sorted + r * a.K;
  const float scale = grad_scale(a.n_norm, T);
  for (int64_t v0 = static_cast<int64_t>(threadIdx.x) * W; v0 < a.ldg; v0 += kGThreads * W) {
    float f[W];
    if (v0 >= a.V) {
#pragma unroll
      for (int j = 0; j < W; ++j) f[j] = 0.f;
    } else {
      const int pb = static_cast<int>(v0 / kPB);
      const float al = salpha[pb];
      GVec<E>::load(row + v0, f);
#pragma unroll
      for (int j = 0; j < W; ++j) f[j] = (v0 + j < a.V) ? f[j] * al : 0.f;
      const int e1 = sboff[pb + 1];
      for (int e = sboff[pb]; e < e1; ++e) {
        const int64_t c = static_cast<int64_t>(__ldg(lidx + e)) - v0;
        if (c >= 0 && c < W) {
          const float sub = __ldg(lp + e) * scale;
#pragma unroll
          for (int j = 0; j < W; ++j)
            if (j == c) f[j] -= sub;
        }
      }
    }
    GVec<E>::store(row + v0, f);
  }
}

// Prepares one chunk's stored exponentials and gathered h for the gradient
// products when every row has one reference (kd_internal.h,
// launch_grad_prepare).  One block per row i < round_up(count, 64).
constexpr int kPrepGradThreads = 128;

__global__ void __launch_bounds__(kPrepGradThreads) grad_prepare_kernel(
    ChunkArgs a, uint16_t* __restrict__ u, uint16_t* __restrict__ hc, int64_t d) {
  const int i = blockIdx.x;
  const int count = chunk_count(a.n_valid, a.row0, a.chunk);
  if (i >= round_up(count, 64)) return;
  uint16_t* row = u + static_cast<int64_t>(i) * a.ldg;
  const int tid = threadIdx.x;
  if (i >= count) {
    // the grad_W product reads whole 64-row blocks: rows past count are zero
    for (int64_t v0 = static_cast<int64_t>(tid) * 8; v0 < a.ldg; v0 += kPrepGradThreads * 8)
      *reinterpret_cast<uint4*>(row + v0) = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  // columns past the last 128-column block, which pass 1 does not write
  for (int64_t v0 = static_cast<int64_t>(a.n_pb) * kPB + tid * 8; v0 < a.ldg;
       v0 += kPrepGradThreads * 8)
    *reinterpret_cast<uint4*>(row + v0) = make_uint4(0u, 0u, 0u, 0u);
  const float ar = a.alpha_row[i];
  if (a.row_flag[i] != 0) {
    // Some blocks of this row kept their own maximum as reference: bring every
    // block to the row's common reference M (a factor 2^(ref_b - M), at most 1).
    const float M = a.mref[i];
    for (int pb = tid; pb < a.n_pb; pb += kPrepGradThreads) {
      const float rb = a.part_m[static_cast<int64_t>(pb) * a.cpad + i];
      if (rb == M) continue;
      const float f = ex2_approx(rb - M);
      uint4* p4 = reinterpret_cast<uint4*>(row + static_cast<int64_t>(pb) * kPB);
#pragma unroll 4
      for (int q = 0; q < kPB / 8; ++q) {
        const uint4 x = p4[q];
        p4[q] = make_uint4(pack_bf16x2(bf16lo_to_f32(x.x) * f, bf16hi_to_f32(x.x) * f),
                           pack_bf16x2(bf16lo_to_f32(x.y) * f, bf16hi_to_f32(x.y) * f),
                           pack_bf16x2(bf16lo_to_f32(x.z) * f, bf16hi_to_f32(x.z) * f),
                           pack_bf16x2(bf16lo_to_f32(x.w) * f, bf16hi_to_f32(x.w) * f));
      }
    }
    __syncthreads();
  }
  {
    // Teacher entries: u[i, v] -= p_v * beta_row, so that alpha_row * u becomes
    // (softmax - p) / (T n).  The sorted list keeps equal indices together:
    // each run is summed first and applied once, by the thread that owns its
    // first entry (distinct runs touch distinct columns).  One entry per
    // thread: its index, its neighbours' and its probability are loaded
    // together, so only the read of u waits on them.
    const float br = a.beta_row[i];
    const int64_t r = a.rows[a.row0 + i];
    const int32_t* lidx = a.idx_sorted + r * a.K;
    const float* lp = a.p_sorted + r * a.K;
    for (int e = tid; e < a.K; e += kPrepGradThreads) {
      const int v = __ldg(lidx + e);
      const int vp = e > 0 ? __ldg(lidx + e - 1) : -1;
      const int vn = e + 1 < a.K ? __ldg(lidx + e + 1) : -1;
      float ps = __ldg(lp + e);
      if (v == kNoIndex || vp == v) continue;
      if (vn == v) {
        ps += __ldg(lp + e + 1);
        for (int f = e + 2; f < a.K && __ldg(lidx + f) == v; ++f) ps += __ldg(lp + f);
      }
      uint16_t* at = row + v;
      const float x = __uint_as_float(static_cast<uint32_t>(*at) << 16);
      *at = static_cast<uint16_t>(pack_bf16x2(fmaf(-ps, br, x), 0.f) & 0xFFFFu);
    }
  }
  // h of this row scaled by alpha_row: grad_W = u^T (alpha_row h)
  uint4* h4 = reinterpret_cast<uint4*>(hc + static_cast<int64_t>(i) * d);
  for (int64_t j = tid; j < d / 8; j += kPrepGradThreads) {
    const uint4 x = h4[j];
    h4[j] = make_uint4(pack_bf16x2(bf16lo_to_f32(x.x) * ar, bf16hi_to_f32(x.x) * ar),
                       pack_bf16x2(bf16lo_to_f32(x.y) * ar, bf16hi_to_f32(x.y) * ar),
                       pack_bf16x2(bf16lo_to_f32(x.z) * ar, bf16hi_to_f32(x.z) * ar),
                       pack_bf16x2(bf16lo_to_f32(x.w) * ar, bf16hi_to_f32(x.w) * ar));
  }
}

// ------------------------------------------------------------- full-vocabulary loss
//
// The teacher distribution is the softmax of the teacher's own logits over the
// whole vocabulary (the pages' online-distillation setting, with nothing
// discarded).  Per row, from the per-block statistics of pass 1 (base-2
// units t2 = z_t log2(e) / T, s2 = z_s log2(e) / T):
//   lse2_t = logsumexp2 of t2, lse2_s = logsumexp2 of s2,
//   sum_v p_v (t2_v - s2_v) = sum_b 2^(m_t,b - lse2_t) a_b,
//   loss_i = ln 2 * (sum_v p_v (t2_v - s2_v) - lse2_t + lse2_s),
// and the factors that turn the stored exponentials into softmax / (T N_valid):
//   alpha_s,b = 2^(m_s,b - lse2_s) / (T N_valid)   (over part_m)
//   alpha_t,b = 2^(m_t,b - lse2_t) / (T N_valid)   (over part_mt).

// row_ok[r] = mask[r] != 0 (every row when there is no mask).
__global__ void mask_rows_kernel(const uint8_t* __restrict__ mask, int64_t N,
                                 int32_t* __restrict__ row_ok) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r < N) row_ok[r] = (mask == nullptr || mask[r] != 0) ? 1 : 0;
}

__device__ __forceinline__ void merge_block(float m, float l, float a, float& M, float& L,
                                            float& A) {
  if (m > M) {
    const float f = ex2_approx(M - m);
    L = L * f + l;
    A = A * f + a;
    M = m;
  } else if (m > -INFINITY) {
    const float f = ex2_approx(m - M);
    L += l * f;
    A += a * f;
  }
}

__global__ void __launch_bounds__(kLseRows * kLseGroups) lse_dual_kernel(
    ChunkArgs a, float* __restrict__ part_mt, const float* __restrict__ part_lt,
    const float* __restrict__ part_a, float T, float* __restrict__ lse_out,
    float* __restrict__ loss_rows) {
  __shared__ float sMt[kLseGroups][kLseRows], sLt[kLseGroups][kLseRows], sA[kLseGroups][kLseRows];
  __shared__ float sMs[kLseGroups][kLseRows], sLs[kLseGroups][kLseRows];
  __shared__ float sLseT[kLseRows], sLseS[kLseRows];
  const int count = chunk_count(a.n_valid, a.row0, a.chunk);
  const int i0 = blockIdx.x * kLseRows;
  if (i0 >= count) return;
  const int x = threadIdx.x, y = threadIdx.y;
  const int i = i0 + x;
  const bool live = i < count;
  float Mt = -INFINITY, Lt = 0.f, At = 0.f, Ms = -INFINITY, Ls = 0.f, dummy = 0.f;
  if (live) {
    // four blocks' statistics loaded before they are merged (same order)
    int pb = y;
    for (; pb + 3 * kLseGroups < a.n_pb; pb += 4 * kLseGroups) {
      float mt[4], lt[4], at[4], ms[4], ls[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t o = static_cast<int64_t>(pb + u * kLseGroups) * a.cpad + i;
        mt[u] = part_mt[o];
        lt[u] = part_lt[o];
        at[u] = part_a[o];
        ms[u] = a.part_m[o];
        ls[u] = a.part_l[o];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        merge_block(mt[u], lt[u], at[u], Mt, Lt, At);
        merge_block(ms[u], ls[u], 0.f, Ms, Ls, dummy);
      }
    }
    for (; pb < a.n_pb; pb += kLseGroups) {
      const int64_t o = static_cast<int64_t>(pb) * a.cpad + i;
      merge_block(part_mt[o], part_lt[o], part_a[o], Mt, Lt, At);
      merge_block(a.part_m[o], a.part_l[o], 0.f, Ms, Ls, dummy);
    }
  }
  sMt[y][x] = Mt;
  sLt[y][x] = Lt;
  sA[y][x] = At;
  sMs[y][x] = Ms;
  sLs[y][x] = Ls;
  __syncthreads();
  if (y == 0 && live) {
    float MT = -INFINITY, LT = 0.f, AT = 0.f, MS = -INFINITY, LS = 0.f;
    for (int g = 0; g < kLseGroups; ++g) {
      merge_block(sMt[g][x], sLt[g][x], sA[g][x], MT, LT, AT);
      merge_block(sMs[g][x], sLs[g][x], 0.f, MS, LS, dummy);
    }
    const float lse2_t = MT + lg2_approx(LT);
    const float lse2_s = MS + lg2_approx(LS);
    const float cross = AT / LT;  // sum_v p_v (t2_v - s2_v)
    loss_rows[a.row0 + i] = kLn2 * (cross - lse2_t + lse2_s);
    lse_out[a.row0 + i] = lse2_s * kLn2;
    sLseT[x] = lse2_t;
    sLseS[x] = lse2_s;
  }
  __syncthreads();
  if (!live) return;
  const float lse2_t = sLseT[x], lse2_s = sLseS[x];
  const float scale = grad_scale(a.n_norm, T);
  int pb = y;
  for (; pb + 3 * kLseGroups < a.n_pb; pb += 4 * kLseGroups) {
    float ms[4], mt[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t o = static_cast<int64_t>(pb + u * kLseGroups) * a.cpad + i;
      ms[u] = a.part_m[o];
      mt[u] = part_mt[o];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t o = static_cast<int64_t>(pb + u * kLseGroups) * a.cpad + i;
      a.part_m[o] = ex2_approx(ms[u] - lse2_s) * scale;
      part_mt[o] = ex2_approx(mt[u] - lse2_t) * scale;
    }
  }
  for (; pb < a.n_pb; pb += kLseGroups) {
    const int64_t o = static_cast<int64_t>(pb) * a.cpad + i;
    a.part_m[o] = ex2_approx(a.part_m[o] - lse2_s) * scale;
    part_mt[o] = ex2_approx(part_mt[o] - lse2_t) * scale;
  }
}

// G[i, v] = u_s[i, v] * alpha_s,b - u_t[i, v] * alpha_t,b (b = v / 128), bf16,
// written over u_s.  Rows count .. round_up(count, 64) and columns >= V are
// zeroed (the grad_W reduction reads whole 64-row blocks).
__global__ void __launch_bounds__(kGThreads) grad_tile_dual_kernel(
    ChunkArgs a, const float* __restrict__ alpha_t, const uint16_t* __restrict__ u_t,
    uint16_t* __restrict__ g) {
  constexpr int W = 8;
  extern __shared__ float sal[];
  float* sas = sal;
  float* sat = sal + a.n_pb;
  const int count = chunk_count(a.n_valid, a.row0, a.chunk);
  const int i = blockIdx.x;
  if (i >= round_up(count, 64)) return;
  uint16_t* row = g + static_cast<int64_t>(i) * a.ldg;
  if (i >= count) {
    float z[W];
#pragma unroll
    for (int j = 0; j < W; ++j) z[j] = 0.f;
    for (int64_t v0 = static_cast<int64_t>(threadIdx.x) * W; v0 < a.ldg; v0 += kGThreads * W)
      GVec<uint16_t>::store(row + v0, z);
    return;
  }
  for (int pb = threadIdx.x; pb < a.n_pb; pb += kGThreads) {
    sas[pb] = a.part_m[static_cast<int64_t>(pb) * a.cpad + i];
    sat[pb] = alpha_t[static_cast<int64_t>(pb) * a.cpad + i];
  }
  __syncthreads();
  const uint16_t* trow = u_t + static_cast<int64_t>(i) * a.ldg;
  for (int64_t v0 = static_cast<int64_t>(threadIdx.x) * W; v0 < a.ldg; v0 += kGThreads * W) {
    float f[W];
    if (v0 >= a.V) {
#pragma unroll
      for (int j = 0; j < W; ++j) f[j] = 0.f;
    } else {
      const int pb = static_cast<int>(v0 / kPB);
      const float as = sas[pb], at = sat[pb];
      float ft[W];
      GVec<uint16_t>::load(row + v0, f);
      GVec<uint16_t>::load(trow + v0, ft);
#pragma unroll
      for (int j = 0; j < W; ++j) f[j] = (v0 + j < a.V) ? fmaf(f[j], as, -ft[j] * at) : 0.f;
    }
    GVec<uint16_t>::store(row + v0, f);
  }
}

// loss = (sum of the per-row terms, in fixed order, in fp64) / n_norm, where
// n_norm is this call's N_valid or that of the whole data-parallel batch.
constexpr int kFinThreads = 1024;

__global__ void __launch_bounds__(kFinThreads) finalize_kernel(const float* __restrict__ loss_rows,
                                                              Ctrl* ctrl,
                                                              const int64_t* __restrict__ n_norm,
                                                              float* loss) {
  __shared__ double sd[kFinThreads];
  const int nv = ctrl->n_valid;
  const int64_t nn = *n_norm;
  double s = 0.0;
  for (int i = threadIdx.x; i < nv; i += kFinThreads) s += static_cast<double>(loss_rows[i]);
  sd[threadIdx.x] = s;
  __syncthreads();
  for (int w = kFinThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) sd[threadIdx.x] += sd[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    ctrl->loss_sum = sd[0];
    *loss = nn > 0 ? static_cast<float>(sd[0] / static_cast<double>(nn)) : 0.f;
  }
}

__global__ void zero_invalid_rows_kernel(const int32_t* __restrict__ row_ok, int64_t d,
                                         float* __restrict__ grad_h) {
  const int64_t r = blockIdx.x;
  if (row_ok[r] != 0) return;
  float* p = grad_h + r * d;
  for (int64_t j = threadIdx.x; j < d; j += blockDim.x) p[j] = 0.f;
}

// ------------------------------------------------------------- fp32 CUDA-core path

// Pass 1 on CUDA cores: a 32-row x 128-column tile of z = h_c W^T in fp32 FMA,
// then the same per-block statistics and stored exponentials as the tensor
// path (fp32 storage; u == nullptr: nothing stored, the loss alone).
constexpr int kSimtRows = 32;
constexpr int kSimtKc = 32;

__global__ void __launch_bounds__(256) simt_pass1_kernel(const float* __restrict__ hc,
                                                        const float* __restrict__ W, int64_t d,
                                                        ChunkArgs a, float k2,
                                                        float* __restrict__ u) {
  __shared__ float sA[kSimtRows][kSimtKc + 1];
  __shared__ float sB[kPB][kSimtKc + 1];
  __shared__ float sZ[kSimtRows][kPB + 1];
  const int count = chunk_count(a.n_valid, a.row0, a.chunk);
  const int i0 = blockIdx.y * kSimtRows;
  if (i0 >= count) return;
  const int pb = blockIdx.x;
  const int col0 = pb * kPB;
  const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
  float acc[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
  for (int64_t k0 = 0; k0 < d; k0 += kSimtKc) {
    for (int e = tid; e < kSimtRows * kSimtKc; e += 256) {
      const int rr = e / kSimtKc, kk = e % kSimtKc;
      const int64_t gi = i0 + rr, gk = k0 + kk;
      sA[rr][kk] = (gi < count && gk < d) ? hc[gi * d + gk] : 0.f;
    }
    for (int e = tid; e < kPB * kSimtKc; e += 256) {
      const int cc = e / kSimtKc, kk = e % kSimtKc;
      const int64_t gv = col0 + cc, gk = k0 + kk;
      sB[cc][kk] = (gv < a.V && gk < d) ? W[gv * d + gk] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < kSimtKc; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) av[r] = sA[ty * 4 + r][kk];
#pragma unroll
      for (int c = 0; c < 4; ++c) bv[c] = sB[tx + 32 * c][kk];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) sZ[ty * 4 + r][tx + 32 * c] = acc[r][c];
  __syncthreads();
  // warp ty handles rows ty*4 .. ty*4+3; lane tx covers columns tx + 32c
  const int nv = min(kPB, a.V - col0);
  for (int r = 0; r < 4; ++r) {
    const int li = ty * 4 + r;
    const int i = i0 + li;
    if (i >= count) break;
    float mx = -INFINITY;
    for (int c = tx; c < nv; c += 32) mx = fmaxf(mx, sZ[li][c]);
    mx = warp_max(mx);
    const float m2 = mx * k2;
    float l = 0.f;
    float* urow = u != nullptr ? u + static_cast<int64_t>(i) * a.ldg + col0 : nullptr;
    for (int c = tx; c < kPB; c += 32) {
      const float e = (c < nv) ? ex2_approx(fmaf(sZ[li][c], k2, -m2)) : 0.f;
      l += e;
      if (urow != nullptr) urow[c] = e;
    }
    l = warp_sum(l);
    float ps = 0.f;
    const int64_t orow = a.rows[a.row0 + i];
    const int lo = a.boff[static_cast<int64_t>(pb) * a.cpad + i];
    const int hi = a.boff[static_cast<int64_t>(pb + 1) * a.cpad + i];
    for (int e = lo + tx; e < hi; e += 32) {
      const int c = (a.idx_sorted[orow * a.K + e] - col0) & (kPB - 1);
      ps += a.p_sorted[orow * a.K + e] * sZ[li][c];
    }
    ps = warp_sum(ps);
    if (tx == 0) {
      const int64_t o = static_cast<int64_t>(pb) * a.cpad + i;
      a.part_m[o] = m2;
      a.part_l[o] = l;
      a.part_ps[o] = ps * k2;
    }
  }
}

// Generic fp32 GEMM on CUDA cores (64 x 64 tiles, 4 x 4 outputs per thread).
constexpr int kGT = 64;
constexpr int kGK = 16;

__global__ void __launch_bounds__(256) simt_gemm_kernel(SimtGemm g) {
  __shared__ float sA[kGK][kGT + 1];
  __shared__ float sB[kGK][kGT + 1];
  int64_t M = g.M_cap, K = g.Kfix;
  if (g.n_valid != nullptr) {
    long long c = static_cast<long long>(*g.n_valid) - g.row0;
    if (c < 0) c = 0;
    if (g.m_from_count) M = c < M ? c : M;
    if (g.k_from_count) K = c < K ? c : K;
  }
  if (K == 0 && g.accumulate) return;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kGT;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kGT;
  if (m0 >= M) return;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  float acc[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
  for (int64_t k0 = 0; k0 < K; k0 += kGK) {
    for (int e = tid; e < kGT * kGK; e += 256) {
      const int kk = e % kGK, mm = e / kGK;
      const int64_t gm = m0 + mm, gk = k0 + kk;
      sA[kk][mm] = (gm < M && gk < K) ? g.A[gm * g.sam + gk * g.sak] : 0.f;
    }
    for (int e = tid; e < kGT * kGK; e += 256) {
      const int nn = e % kGT, kk = e / kGT;
      const int64_t gn = n0 + nn, gk = k0 + kk;
      sB[kk][nn] = (gn < g.N && gk < K) ? g.B[gk * g.sbk + gn * g.sbn] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kGK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) av[r] = sA[kk][ty * 4 + r];
#pragma unroll
      for (int c = 0; c < 4; ++c) bv[c] = sB[kk][tx + 16 * c];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int64_t gm = m0 + ty * 4 + r;
    if (gm >= M) continue;
    const int64_t orow = g.row_map != nullptr ? g.row_map[g.row_map_off + gm] : gm;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int64_t gn = n0 + tx + 16 * c;
      if (gn >= g.N) continue;
      float* p = g.C + orow * g.ldc + gn;
      *p = g.accumulate ? *p + acc[r][c] : acc[r][c];
    }
  }
}

int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

}  // namespace

// ------------------------------------------------------------------ launchers

cudaError_t launch_teacher_prep(const int32_t* idx, const float* logit, const uint8_t* mask,
                                int64_t N, int K, int64_t V, float T, int32_t* row_ok,
                                int32_t* idx_sorted, float* p_sorted, float* plogp, float* psum,
                                int32_t* top1, uint32_t* err, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  const int P2 = next_pow2(K < 2 ? 2 : K);
  if (P2 <= 128) {
    // one warp per row, the entries in registers
    const unsigned grid = static_cast<unsigned>(ceil_div(N, kPrepWarpRows));
    const float k2 = kLog2e / T;
    if (P2 <= 32)
      teacher_prep_warp_kernel<1><<<grid, 32 * kPrepWarpRows, 0, s>>>(
          idx, logit, mask, N, K, V, k2, row_ok, idx_sorted, p_sorted, plogp, psum, top1, err);
    else if (P2 == 64)
      teacher_prep_warp_kernel<2><<<grid, 32 * kPrepWarpRows, 0, s>>>(
          idx, logit, mask, N, K, V, k2, row_ok, idx_sorted, p_sorted, plogp, psum, top1, err);
    else
      teacher_prep_warp_kernel<4><<<grid, 32 * kPrepWarpRows, 0, s>>>(
          idx, logit, mask, N, K, V, k2, row_ok, idx_sorted, p_sorted, plogp, psum, top1, err);
    return cudaGetLastError();
  }
  const size_t smem = static_cast<size_t>(P2) * 8;
  cudaError_t e = cudaFuncSetAttribute(teacher_prep_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem < 48 * 1024 ? 48 * 1024 : smem));
  if (e != cudaSuccess) return e;
  teacher_prep_kernel<<<static_cast<unsigned>(N), kPrepThreads, smem, s>>>(
      idx, logit, mask, K, V, kLog2e / T, P2, row_ok, idx_sorted, p_sorted, plogp, psum, top1,
      err);
  return cudaGetLastError();
}

cudaError_t launch_compact(const int32_t* row_ok, int64_t N, int32_t* rows, Ctrl* ctrl,
                           int64_t* n_valid_out, cudaStream_t s) {
  compact_kernel<<<1, kScanThreads, 0, s>>>(row_ok, N, rows, ctrl, n_valid_out);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void* h, size_t elem, int64_t d, const ChunkArgs& a,
                               void* hc, const void* W, const int32_t* top1, float k2,
                               cudaStream_t s) {
  if (a.mref != nullptr && (elem != 2 || W == nullptr || top1 == nullptr))
    return cudaErrorInvalidValue;
  gather_rows_kernel<<<static_cast<unsigned>(round_up(a.chunk, 128)), kGatherThreads, 0, s>>>(
      static_cast<const uint8_t*>(h), d * static_cast<int64_t>(elem), a,
      static_cast<uint8_t*>(hc), static_cast<const uint8_t*>(W), top1, k2);
  return cudaGetLastError();
}

cudaError_t launch_grad_prepare(const ChunkArgs& a, uint16_t* u, uint16_t* hc, int64_t d,
                                cudaStream_t s) {
  if (a.alpha_row == nullptr || d % 8 != 0) return cudaErrorInvalidValue;
  grad_prepare_kernel<<<static_cast<unsigned>(round_up(a.chunk, 64)), kPrepGradThreads, 0, s>>>(
      a, u, hc, d);
  return cudaGetLastError();
}

cudaError_t launch_bucket_offsets(const ChunkArgs& a, cudaStream_t s) {
  const dim3 block(kBoffRows, kBoffGroups);
  const dim3 grid(static_cast<unsigned>(ceil_div(a.chunk, kBoffRows)),
                  static_cast<unsigned>(ceil_div(a.n_pb + 1, kBoffGroups * kBoffPerThread)));
  bucket_offsets_kernel<<<grid, block, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_lse(const ChunkArgs& a, const float* plogp, const float* psum, float T,
                       float* lse, float* loss_rows, cudaStream_t s) {
  const dim3 block(kLseRows, kLseGroups);
  lse_kernel<<<static_cast<unsigned>(ceil_div(a.chunk, kLseRows)), block, 0, s>>>(
      a, plogp, psum, T, lse, loss_rows);
  return cudaGetLastError();
}

cudaError_t launch_grad_tile(const ChunkArgs& a, void* g, size_t elem, float T, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(a.n_pb) * 4 + static_cast<size_t>(a.n_pb + 1) * 2 + 16;
  const unsigned grid = static_cast<unsigned>(round_up(a.chunk, 64));
  cudaError_t e;
  if (elem == 2) {
    e = cudaFuncSetAttribute(grad_tile_kernel<uint16_t>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem < 48 * 1024 ? 48 * 1024 : smem));
    if (e != cudaSuccess) return e;
    grad_tile_kernel<uint16_t><<<grid, kGThreads, smem, s>>>(a, static_cast<uint16_t*>(g), T);
  } else {
    e = cudaFuncSetAttribute(grad_tile_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem < 48 * 1024 ? 48 * 1024 : smem));
    if (e != cudaSuccess) return e;
    grad_tile_kernel<float><<<grid, kGThreads, smem, s>>>(a, static_cast<float*>(g), T);
  }
  return cudaGetLastError();
}

cudaError_t launch_finalize(const float* loss_rows, Ctrl* ctrl, const int64_t* n_norm,
                            float* loss, cudaStream_t s) {
  finalize_kernel<<<1, kFinThreads, 0, s>>>(loss_rows, ctrl, n_norm, loss);
  return cudaGetLastError();
}

cudaError_t launch_zero_invalid_rows(const int32_t* row_ok, int64_t N, int64_t d, float* grad_h,
                                     cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  zero_invalid_rows_kernel<<<static_cast<unsigned>(N), 128, 0, s>>>(row_ok, d, grad_h);
  return cudaGetLastError();
}

cudaError_t launch_simt_pass1(const float* hc, const float* W, int64_t d, const ChunkArgs& a,
                              float k2, float* u, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(a.n_pb), static_cast<unsigned>(ceil_div(a.chunk, kSimtRows)));
  simt_pass1_kernel<<<grid, 256, 0, s>>>(hc, W, d, a, k2, u);
  return cudaGetLastError();
}

cudaError_t launch_simt_gemm(const SimtGemm& g, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(ceil_div(g.N, kGT)),
                  static_cast<unsigned>(ceil_div(g.M_cap, kGT)));
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  simt_gemm_kernel<<<grid, 256, 0, s>>>(g);
  return cudaGetLastError();
}

cudaError_t launch_mask_rows(const uint8_t* mask, int64_t N, int32_t* row_ok, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  mask_rows_kernel<<<static_cast<unsigned>(ceil_div(N, 256)), 256, 0, s>>>(mask, N, row_ok);
  return cudaGetLastError();
}

cudaError_t launch_lse_dual(const ChunkArgs& a, float* part_mt, const float* part_lt,
                            const float* part_a, float T, float* lse, float* loss_rows,
                            cudaStream_t s) {
  const dim3 block(kLseRows, kLseGroups);
  lse_dual_kernel<<<static_cast<unsigned>(ceil_div(a.chunk, kLseRows)), block, 0, s>>>(
      a, part_mt, part_lt, part_a, T, lse, loss_rows);
  return cudaGetLastError();
}

cudaError_t launch_grad_tile_dual(const ChunkArgs& a, const float* alpha_t, const uint16_t* u_t,
                                  uint16_t* g, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(a.n_pb) * 8 + 16;
  cudaError_t e = cudaFuncSetAttribute(grad_tile_dual_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem < 48 * 1024 ? 48 * 1024 : smem));
  if (e != cudaSuccess) return e;
  grad_tile_dual_kernel<<<static_cast<unsigned>(round_up(a.chunk, 64)), kGThreads, smem, s>>>(
      a, alpha_t, u_t, g);
  return cudaGetLastError();
}

}  // namespace kd
