// hpa_decode_attn_combine_noalloc: split-KV attention + combine for callers
// that cannot allocate device memory.
//
// The split partials (per-segment o and lse) normally live in buffers the
// caller allocates.  Some callers cannot do that on the decode path: a
// plugin running inside another runtime that owns the whole device memory
// pool and hands out no workspace, or a serving loop that must not call
// cudaMalloc/cudaFree mid-step (cudaFree synchronises the device, and either
// call can fail under memory pressure).  For them, the partials live in the
// fixed array below, which is part of this library's device image: every GPU
// that loads it holds the array until the process exits.
//
// Set-up: in host code the array's name is only a host-side stand-in, so the
// first call in each CUDA context (normally once per device: the runtime's
// primary context) resolves the array's device address with
// cudaGetSymbolAddress while that context is current; that may also load this
// module.  The first call should therefore come before any stream capture.
// The address is cached under the context's process-unique id, so a caller
// that switches to a context of its own, or a new primary context after
// cudaDeviceReset, gets that context's address, never a stale one.
//
// Every call shares the one array, so calls that overlap on the GPU
// (different streams, or several host threads) race on it; serialise them.
// Nothing in the array needs to start at zero: the attention kernel writes
// every partial row the combine kernel reads in the same call, so rows left
// by an earlier, larger call are never read.
#include <cudaTypedefs.h>

#include <mutex>

#include "hpa_internal.cuh"

namespace {

constexpr size_t kScratchFloats = HPA_NOALLOC_SCRATCH_BYTES / sizeof(float);
static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

// ---- the current context's unique id (driver API, reached through the runtime)
struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const CtxFns &ctx_fns() {
  static CtxFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  return fns;
}

// Unique id of the current context, or 0 when there is none yet (or it cannot be read).
unsigned long long current_ctx_id() {
  const CtxFns &f = ctx_fns();
  if (!f.get_current || !f.get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (f.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

constexpr int kCacheEntries = 64;
std::mutex g_mu;
unsigned long long g_ids[kCacheEntries] = {0};
float *g_ptrs[kCacheEntries] = {nullptr};
int g_next = 0;

// Device address of the array in the current context.
cudaError_t scratch_address(float **out) {
  unsigned long long id = current_ctx_id();
  if (id != 0) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < kCacheEntries; ++i)
      if (g_ids[i] == id) {
        *out = g_ptrs[i];
        return cudaSuccess;
      }
  }
  void *p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // set-up for this context
  if (e != cudaSuccess) return e;
  *out = static_cast<float *>(p);
  if (id == 0) id = current_ctx_id();  // the runtime may have just made its primary context
  if (id != 0) {                        // no id readable: look the address up on every call
    std::lock_guard<std::mutex> lk(g_mu);
    g_ids[g_next] = id;
    g_ptrs[g_next] = *out;
    g_next = (g_next + 1) % kCacheEntries;
  }
  return cudaSuccess;
}

}  // namespace

extern "C" int hpa_decode_attn_combine_noalloc(
    const void *q_dev, const void *k_pool_dev, const void *v_pool_dev, int32_t kv_dtype,
    const float *k_scale_dev, const float *v_scale_dev, int64_t num_pages,
    const int32_t *page_indptr_dev, const int32_t *page_indices_dev, int32_t page_size,
    int32_t B, int32_t q_len, int32_t Hq, int32_t Hkv, int32_t d, float sm_scale,
    void *taskmap_dev, int32_t num_ctas, void *out_dev, float *out_lse_dev,
    hpa_stream_t stream) {
  const int32_t cap = hpa_max_segments(B, num_ctas);
  if (cap <= 0 || q_len < 1 || Hq < 1 || d < 1) return HPA_ERR_INVALID;
  // partial_o rows are d floats, partial_lse rows one float; partial_o comes first,
  // so partial_lse starts 16-byte aligned whenever d is a multiple of 4.
  const int64_t rows = int64_t(cap) * q_len * Hq;
  const int64_t o_floats = rows * d;
  if (o_floats + rows > static_cast<int64_t>(kScratchFloats)) return HPA_ERR_NOALLOC_CAPACITY;
  float *scratch = nullptr;
  const cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    cudaGetLastError();  // the failed lookup is reported here, not left for the caller's next check
    return hpa::cuda_fail(e);
  }
  int rc = hpa_decode_attn(q_dev, k_pool_dev, v_pool_dev, kv_dtype, k_scale_dev, v_scale_dev,
                           num_pages, page_indptr_dev, page_indices_dev, page_size, B, q_len,
                           Hq, Hkv, d, sm_scale, taskmap_dev, num_ctas, scratch,
                           scratch + o_floats, stream);
  if (rc != HPA_OK) return rc;
  return hpa_combine(scratch, scratch + o_floats, taskmap_dev, B, num_ctas, q_len, Hq, d,
                     out_dev, out_lse_dev, stream);
}
