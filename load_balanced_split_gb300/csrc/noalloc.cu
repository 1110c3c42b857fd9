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
// The set-up is done by the first call on each device: with that device
// current, cudaGetSymbolAddress resolves the array's device address (which
// also loads this module if it is not loaded yet).  That first call should
// therefore come before any stream capture.  Every call shares the one array,
// so calls that overlap on the GPU (different streams, or several host
// threads) race on it; serialise them.  Nothing in the array needs to start
// at zero: the attention kernel writes every partial row the combine kernel
// reads in the same call, so stale contents from an earlier call are never
// read.
#include <mutex>

#include "hpa_internal.cuh"

namespace {

constexpr size_t kScratchFloats = HPA_NOALLOC_SCRATCH_BYTES / sizeof(float);
static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the array on the current device (resolved once per device).
cudaError_t scratch_for_current_device(float **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<float *>(p);
  }
  *out = g_scratch_ptr[dev];
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
  cudaError_t e = scratch_for_current_device(&scratch);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return HPA_ERR_CUDA;
  }
  int rc = hpa_decode_attn(q_dev, k_pool_dev, v_pool_dev, kv_dtype, k_scale_dev, v_scale_dev,
                           num_pages, page_indptr_dev, page_indices_dev, page_size, B, q_len,
                           Hq, Hkv, d, sm_scale, taskmap_dev, num_ctas, scratch,
                           scratch + o_floats, stream);
  if (rc != HPA_OK) return rc;
  return hpa_combine(scratch, scratch + o_floats, taskmap_dev, B, num_ctas, q_len, Hq, d,
                     out_dev, out_lse_dev, stream);
}
