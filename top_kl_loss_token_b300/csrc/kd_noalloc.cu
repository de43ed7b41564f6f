// kd_noalloc.cu -- kd_topk_kl_fwd_bwd_noalloc: the fused fwd+bwd call with its
// workspace in a fixed device array that the library owns, for callers that
// cannot allocate device memory themselves.
//
// Some callers can't call cudaMalloc: processes whose caching allocator owns
// the device memory and forbids raw cudaMalloc beside its pool, and plug-ins
// or embedded runtimes that are handed device pointers for their inputs and
// outputs but no allocator.  This entry point lets them run the loss anyway,
// up to a fixed size.
//
// The scratch array is a file-scope __device__ array; in host code its name is
// only a stand-in, so its device address is looked up with
// cudaGetSymbolAddress once per device (with that device current) and that
// address is what the kernels receive.
#include <mutex>

#include "kd_internal.h"

namespace {

static __device__ __align__(256) unsigned char kd_noalloc_scratch[KD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up on the
// first call made with that device current.  nullptr on failure.
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, kd_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // consume the error so a later, unrelated call does not report it
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

bool fits(int64_t N, int64_t d, int64_t V, int32_t K, int64_t chunk, kd_dtype dtype) {
  const size_t need = kd_topk_kl_workspace_bytes(N, d, V, K, chunk, dtype);
  return need != 0 && need <= static_cast<size_t>(KD_NOALLOC_SCRATCH_BYTES);
}

}  // namespace

extern "C" kd_status kd_topk_kl_fwd_bwd_noalloc(const void* h, const void* W, kd_dtype dtype,
                                                const int32_t* topk_idx,
                                                const float* topk_logit, const uint8_t* mask,
                                                int64_t N, int64_t d, int64_t V, int32_t K,
                                                float T, int64_t chunk, float* loss,
                                                float* grad_h, float* grad_W,
                                                uint32_t* dev_err_flags, cudaStream_t stream) {
  // Sizes first, on the host only: a request that cannot fit is rejected
  // before any CUDA call.
  kd::Plan plan;
  const kd_status st = kd::make_plan(N, d, V, K, chunk > 0 ? chunk : 128, dtype, &plan);
  if (st != KD_OK) return st;
  int64_t c = chunk;
  if (c > 0) {
    if (!fits(N, d, V, K, c, dtype)) return KD_ERR_WORKSPACE;
  } else {
    // The largest multiple of 128 tokens, up to the default chunk, whose
    // workspace fits (the workspace grows with the chunk).
    const int64_t hi_c = kd_topk_kl_default_chunk(N, d, V, dtype);
    if (!fits(N, d, V, K, 128, dtype)) return KD_ERR_WORKSPACE;
    int64_t lo = 1, hi = hi_c / 128;  // in units of 128 tokens; lo always fits
    while (lo < hi) {
      const int64_t mid = (lo + hi + 1) / 2;
      if (fits(N, d, V, K, mid * 128, dtype)) lo = mid;
      else hi = mid - 1;
    }
    c = lo * 128;
  }
  void* ws = scratch_address();
  if (ws == nullptr) return KD_ERR_CUDA;
  return kd_topk_kl_fwd_bwd(h, W, dtype, topk_idx, topk_logit, mask, N, d, V, K, T, c, loss,
                            grad_h, grad_W, ws, KD_NOALLOC_SCRATCH_BYTES, dev_err_flags, stream);
}
