// C ABI of libhpa: argument checks, task map sizing, TMA descriptor set-up
// and kernel launches.  See include/hpa.h for the contract of every call.
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>

#include "hpa_internal.cuh"

namespace hpa {

namespace {
thread_local int g_last_cuda_error = 0;  // what hpa_last_cuda_error() reports, per thread
}  // namespace

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return HPA_ERR_CUDA;
}

int last_cuda_error() { return g_last_cuda_error; }

}  // namespace hpa

namespace {

using hpa::cuda_fail;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int32_t kMaxB = 1 << 24;
constexpr int32_t kMaxC = 1 << 20;

int64_t taskmap_words(int64_t B, int64_t C, int64_t s_cap) {
  return hpa::TaskMapLayout::make(B, C).words(s_cap);
}

// ---- TMA descriptors for a KV pool: 3-D view (d, token-in-page, page*Hkv + head)
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

struct MapKey {
  const void *ptr;
  int64_t rows;
  int kv_dtype;
  bool operator==(const MapKey &o) const {
    return ptr == o.ptr && rows == o.rows && kv_dtype == o.kv_dtype;
  }
};

std::mutex g_map_mu;
constexpr int kMapCache = 8;
MapKey g_map_keys[kMapCache];
CUtensorMap g_maps[kMapCache];
int g_map_next = 0, g_map_used = 0;

int pool_map(const void *pool, int64_t num_pages, int Hkv, int kv_dtype, CUtensorMap *out) {
  const int64_t zdim = num_pages * Hkv;
  const MapKey key{pool, zdim, kv_dtype};
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    for (int i = 0; i < g_map_used; ++i)
      if (g_map_keys[i] == key) {
        *out = g_maps[i];
        return HPA_OK;
      }
  }
  auto fn = encode_fn();
  if (!fn) return cuda_fail(cudaErrorNotSupported);
  const int es = kv_dtype == HPA_KV_BF16 ? 2 : 1;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(hpa::HEAD_DIM),
                              static_cast<cuuint64_t>(hpa::PAGE), static_cast<cuuint64_t>(zdim)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(hpa::HEAD_DIM * es),
                                 static_cast<cuuint64_t>(hpa::HEAD_DIM * es * hpa::PAGE)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), static_cast<cuuint32_t>(hpa::PAGE),
                             1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  CUtensorMap m;
  CUresult r = fn(&m,
                  kv_dtype == HPA_KV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                          : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                  3, const_cast<void *>(pool), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return HPA_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_map_mu);
  g_map_keys[g_map_next] = key;
  g_maps[g_map_next] = m;
  g_map_next = (g_map_next + 1) % kMapCache;
  if (g_map_used < kMapCache) ++g_map_used;
  *out = m;
  return HPA_OK;
}

int check_plan_args(const int32_t *seq_lens, int32_t B, int32_t tile, int64_t C,
                    const void *tm, size_t bytes, int64_t s_cap) {
  if (!seq_lens || !tm) return HPA_ERR_INVALID;
  if (B < 1 || B > kMaxB || C < 1 || C > kMaxC) return HPA_ERR_INVALID;
  if (tile < hpa::PAGE || tile % hpa::PAGE != 0) return HPA_ERR_INVALID;
  if (!aligned(tm, 16)) return HPA_ERR_ALIGN;
  if (bytes < static_cast<size_t>(taskmap_words(B, C, s_cap)) * 4) return HPA_ERR_WORKSPACE;
  return HPA_OK;
}

}  // namespace

extern "C" {

size_t hpa_taskmap_bytes(int32_t B, int32_t num_ctas) {
  if (B < 1 || B > kMaxB || num_ctas < 1 || num_ctas > kMaxC) return 0;
  return static_cast<size_t>(taskmap_words(B, num_ctas, int64_t(B) + num_ctas - 1)) * 4;
}

int32_t hpa_max_segments(int32_t B, int32_t num_ctas) {
  if (B < 1 || B > kMaxB || num_ctas < 1 || num_ctas > kMaxC) return 0;
  return B + num_ctas - 1;
}

int32_t hpa_static_num_ctas(int32_t B, int32_t splits) {
  if (B < 1 || B > kMaxB || splits < 1 || int64_t(B) * splits > kMaxC) return 0;
  return B * splits;
}

size_t hpa_static_taskmap_bytes(int32_t B, int32_t splits) {
  const int32_t C = hpa_static_num_ctas(B, splits);
  if (C == 0) return 0;
  return static_cast<size_t>(taskmap_words(B, C, C)) * 4;
}

int32_t hpa_default_num_ctas_mma(int32_t Hq, int32_t Hkv, int32_t q_len, int32_t kv_dtype) {
  if (Hkv < 1 || Hq < Hkv || Hq % Hkv != 0 || q_len < 1 ||
      (kv_dtype != HPA_KV_BF16 && kv_dtype != HPA_KV_E4M3))
    return -1;
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    cuda_fail(e);
    return -1;
  }
  if (hpa::attn_ctas_per_sm(kv_dtype, q_len, &per_sm) != 0 || per_sm < 1) return -1;
  // one CTA per (partition, KV head, group of 16 query rows)
  const int groups = ((Hq / Hkv) * q_len + hpa::MAX_ROWS - 1) / hpa::MAX_ROWS;
  const int c = sms * per_sm / (Hkv * groups);
  return c < 1 ? 1 : c;
}

int hpa_plan(const int32_t *seq_lens_dev, int32_t B, int32_t tile, int32_t num_ctas,
             void *taskmap_dev, size_t taskmap_bytes, hpa_stream_t stream) {
  const int64_t s_cap = int64_t(B) + num_ctas - 1;
  int rc = check_plan_args(seq_lens_dev, B, tile, num_ctas, taskmap_dev, taskmap_bytes, s_cap);
  if (rc != HPA_OK) return rc;
  cudaError_t e = hpa::launch_plan(seq_lens_dev, B, tile, num_ctas, 0, 0,
                                   static_cast<int32_t *>(taskmap_dev), s_cap,
                                   reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? HPA_OK : cuda_fail(e);
}

int hpa_plan_weighted(const int32_t *seq_lens_dev, int32_t B, int32_t tile, int32_t num_ctas,
                      void *taskmap_dev, size_t taskmap_bytes, hpa_stream_t stream) {
  const int64_t s_cap = int64_t(B) + num_ctas - 1;
  int rc = check_plan_args(seq_lens_dev, B, tile, num_ctas, taskmap_dev, taskmap_bytes, s_cap);
  if (rc != HPA_OK) return rc;
  if (hpa::plan_stage_bytes(B, num_ctas, 2) > hpa::kPlanStageLimit) return HPA_ERR_UNSUPPORTED;
  cudaError_t e = hpa::launch_plan(seq_lens_dev, B, tile, num_ctas, 2, 0,
                                   static_cast<int32_t *>(taskmap_dev), s_cap,
                                   reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? HPA_OK : cuda_fail(e);
}

int hpa_plan_static(const int32_t *seq_lens_dev, int32_t B, int32_t tile, int32_t splits,
                    void *taskmap_dev, size_t taskmap_bytes, hpa_stream_t stream) {
  const int32_t C = hpa_static_num_ctas(B, splits);
  if (C == 0) return HPA_ERR_INVALID;
  int rc = check_plan_args(seq_lens_dev, B, tile, C, taskmap_dev, taskmap_bytes, C);
  if (rc != HPA_OK) return rc;
  cudaError_t e = hpa::launch_plan(seq_lens_dev, B, tile, C, 1, splits,
                                   static_cast<int32_t *>(taskmap_dev), C,
                                   reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? HPA_OK : cuda_fail(e);
}

static int decode_attn_impl(const void *q_dev, const void *k_pool_dev, const void *v_pool_dev,
                            int32_t kv_dtype, const float *k_scale_dev,
                            const float *v_scale_dev, int64_t num_pages,
                            const int32_t *page_indptr_dev, const int32_t *page_indices_dev,
                            int32_t page_size, int32_t B, int32_t q_len, int32_t Hq, int32_t Hkv,
                            int32_t d, float sm_scale, void *taskmap_dev, int32_t num_ctas,
                            float *partial_o_dev, float *partial_lse_dev, uint64_t *trace_dev,
                            void *out_dev, float *out_lse_dev, int32_t *arrivals_dev,
                            hpa_stream_t stream, bool tc = false, bool all_heads = false) {
  if (!q_dev || !k_pool_dev || !v_pool_dev || !page_indptr_dev || !page_indices_dev ||
      !taskmap_dev || !partial_o_dev || !partial_lse_dev)
    return HPA_ERR_INVALID;
  if (kv_dtype != HPA_KV_BF16 && kv_dtype != HPA_KV_E4M3) return HPA_ERR_INVALID;
  if (kv_dtype == HPA_KV_E4M3 && (!k_scale_dev || !v_scale_dev)) return HPA_ERR_INVALID;
  if (B < 1 || B > kMaxB || num_ctas < 1 || num_ctas > kMaxC || q_len < 1 || Hq < 1 ||
      Hkv < 1 || Hkv > 65535 || num_pages < 1 || !std::isfinite(sm_scale))
    return HPA_ERR_INVALID;
  if (d != hpa::HEAD_DIM || page_size != hpa::PAGE || Hq % Hkv != 0 ||
      int64_t(Hq / Hkv) * q_len > hpa::MAX_ROWS_TOTAL)
    return HPA_ERR_UNSUPPORTED;
  if (num_pages * Hkv > INT_MAX) return HPA_ERR_UNSUPPORTED;
  if (!aligned(q_dev, 16) || !aligned(k_pool_dev, 16) || !aligned(v_pool_dev, 16) ||
      !aligned(taskmap_dev, 16) || !aligned(partial_o_dev, 16) || !aligned(partial_lse_dev, 4))
    return HPA_ERR_ALIGN;
  CUtensorMap tmk, tmv;
  int rc = pool_map(k_pool_dev, num_pages, Hkv, kv_dtype, &tmk);
  if (rc == HPA_OK) rc = pool_map(v_pool_dev, num_pages, Hkv, kv_dtype, &tmv);
  if (rc != HPA_OK) return rc;
  hpa::AttnParams p;
  p.q = static_cast<const __nv_bfloat16 *>(q_dev);
  p.tm = static_cast<int32_t *>(taskmap_dev);
  p.page_indptr = page_indptr_dev;
  p.page_indices = page_indices_dev;
  p.k_scale = k_scale_dev;
  p.v_scale = v_scale_dev;
  p.partial_o = partial_o_dev;
  p.partial_lse = partial_lse_dev;
  p.trace = reinterpret_cast<unsigned long long *>(trace_dev);
  p.out = static_cast<__nv_bfloat16 *>(out_dev);
  p.out_lse = out_lse_dev;
  p.arrivals = arrivals_dev;
  p.num_pages = num_pages;
  p.lay = hpa::TaskMapLayout::make(B, num_ctas);
  p.B = B;
  p.C = num_ctas;
  p.q_len = q_len;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.rows = p.G * q_len;
  p.heads_per_cta = all_heads ? Hkv : 1;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  cudaError_t e =
      tc ? hpa::launch_decode_attn_tc(p, tmk, tmv, kv_dtype, reinterpret_cast<cudaStream_t>(stream))
         : hpa::launch_decode_attn(p, tmk, tmv, kv_dtype, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? HPA_OK : cuda_fail(e);
}

int hpa_decode_attn_tc(const void *q_dev, const void *k_pool_dev, const void *v_pool_dev,
                       int32_t kv_dtype, const float *k_scale_dev, const float *v_scale_dev,
                       int64_t num_pages, const int32_t *page_indptr_dev,
                       const int32_t *page_indices_dev, int32_t page_size, int32_t B,
                       int32_t q_len, int32_t Hq, int32_t Hkv, int32_t d, float sm_scale,
                       void *taskmap_dev, int32_t num_ctas, float *partial_o_dev,
                       float *partial_lse_dev, hpa_stream_t stream) {
  return decode_attn_impl(q_dev, k_pool_dev, v_pool_dev, kv_dtype, k_scale_dev, v_scale_dev,
                          num_pages, page_indptr_dev, page_indices_dev, page_size, B, q_len, Hq,
                          Hkv, d, sm_scale, taskmap_dev, num_ctas, partial_o_dev,
                          partial_lse_dev, nullptr, nullptr, nullptr, nullptr, stream, true);
}

int32_t hpa_default_num_ctas_tc(int32_t Hq, int32_t Hkv, int32_t q_len, int32_t kv_dtype) {
  if (Hkv < 1 || Hq < Hkv || Hq % Hkv != 0 || q_len < 1 ||
      int64_t(Hq / Hkv) * q_len > hpa::MAX_ROWS_TOTAL ||
      (kv_dtype != HPA_KV_BF16 && kv_dtype != HPA_KV_E4M3))
    return -1;
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    cuda_fail(e);
    return -1;
  }
  if (hpa::attn_tc_ctas_per_sm(kv_dtype, (Hq / Hkv) * q_len, &per_sm) != 0 || per_sm < 1)
    return -1;
  const int c = sms * per_sm / Hkv;
  return c < 1 ? 1 : c;
}

int hpa_decode_attn_mma(const void *q_dev, const void *k_pool_dev, const void *v_pool_dev,
                        int32_t kv_dtype, const float *k_scale_dev, const float *v_scale_dev,
                        int64_t num_pages, const int32_t *page_indptr_dev,
                        const int32_t *page_indices_dev, int32_t page_size, int32_t B,
                        int32_t q_len, int32_t Hq, int32_t Hkv, int32_t d, float sm_scale,
                        void *taskmap_dev, int32_t num_ctas, float *partial_o_dev,
                        float *partial_lse_dev, hpa_stream_t stream) {
  return decode_attn_impl(q_dev, k_pool_dev, v_pool_dev, kv_dtype, k_scale_dev, v_scale_dev,
                          num_pages, page_indptr_dev, page_indices_dev, page_size, B, q_len, Hq,
                          Hkv, d, sm_scale, taskmap_dev, num_ctas, partial_o_dev,
                          partial_lse_dev, nullptr, nullptr, nullptr, nullptr, stream);
}

// More than 16 query rows per KV head (MTP with several draft tokens) go to the
// tcgen05 kernel, which takes all rows in one pass over the keys.
static bool routes_to_tc(int32_t Hq, int32_t Hkv, int32_t q_len) {
  return Hkv >= 1 && Hq % Hkv == 0 && int64_t(Hq / Hkv) * q_len > hpa::MAX_ROWS;
}

int hpa_decode_attn(const void *q_dev, const void *k_pool_dev, const void *v_pool_dev,
                    int32_t kv_dtype, const float *k_scale_dev, const float *v_scale_dev,
                    int64_t num_pages, const int32_t *page_indptr_dev,
                    const int32_t *page_indices_dev, int32_t page_size, int32_t B,
                    int32_t q_len, int32_t Hq, int32_t Hkv, int32_t d, float sm_scale,
                    void *taskmap_dev, int32_t num_ctas, float *partial_o_dev,
                    float *partial_lse_dev, hpa_stream_t stream) {
  return decode_attn_impl(q_dev, k_pool_dev, v_pool_dev, kv_dtype, k_scale_dev, v_scale_dev,
                          num_pages, page_indptr_dev, page_indices_dev, page_size, B, q_len, Hq,
                          Hkv, d, sm_scale, taskmap_dev, num_ctas, partial_o_dev,
                          partial_lse_dev, nullptr, nullptr, nullptr, nullptr, stream,
                          routes_to_tc(Hq, Hkv, q_len));
}

int32_t hpa_default_num_ctas(int32_t Hq, int32_t Hkv, int32_t q_len, int32_t kv_dtype) {
  return routes_to_tc(Hq, Hkv, q_len) ? hpa_default_num_ctas_tc(Hq, Hkv, q_len, kv_dtype)
                                      : hpa_default_num_ctas_mma(Hq, Hkv, q_len, kv_dtype);
}

int hpa_decode_attn_traced(const void *q_dev, const void *k_pool_dev, const void *v_pool_dev,
                           int32_t kv_dtype, const float *k_scale_dev, const float *v_scale_dev,
                           int64_t num_pages, const int32_t *page_indptr_dev,
                           const int32_t *page_indices_dev, int32_t page_size, int32_t B,
                           int32_t q_len, int32_t Hq, int32_t Hkv, int32_t d, float sm_scale,
                           void *taskmap_dev, int32_t num_ctas, float *partial_o_dev,
                           float *partial_lse_dev, uint64_t *trace_dev, hpa_stream_t stream) {
  if (!trace_dev) return HPA_ERR_INVALID;
  if (!aligned(trace_dev, 8)) return HPA_ERR_ALIGN;
  return decode_attn_impl(q_dev, k_pool_dev, v_pool_dev, kv_dtype, k_scale_dev, v_scale_dev,
                          num_pages, page_indptr_dev, page_indices_dev, page_size, B, q_len, Hq,
                          Hkv, d, sm_scale, taskmap_dev, num_ctas, partial_o_dev,
                          partial_lse_dev, trace_dev, nullptr, nullptr, nullptr, stream,
                          routes_to_tc(Hq, Hkv, q_len));
}

int hpa_decode_attn_allheads(const void *q_dev, const void *k_pool_dev, const void *v_pool_dev,
                             int32_t kv_dtype, const float *k_scale_dev,
                             const float *v_scale_dev, int64_t num_pages,
                             const int32_t *page_indptr_dev, const int32_t *page_indices_dev,
                             int32_t page_size, int32_t B, int32_t q_len, int32_t Hq,
                             int32_t Hkv, int32_t d, float sm_scale, void *taskmap_dev,
                             int32_t num_ctas, float *partial_o_dev, float *partial_lse_dev,
                             uint64_t *trace_dev, hpa_stream_t stream) {
  if (trace_dev && !aligned(trace_dev, 8)) return HPA_ERR_ALIGN;
  return decode_attn_impl(q_dev, k_pool_dev, v_pool_dev, kv_dtype, k_scale_dev, v_scale_dev,
                          num_pages, page_indptr_dev, page_indices_dev, page_size, B, q_len, Hq,
                          Hkv, d, sm_scale, taskmap_dev, num_ctas, partial_o_dev,
                          partial_lse_dev, trace_dev, nullptr, nullptr, nullptr, stream, false,
                          true);
}

int32_t hpa_default_num_ctas_allheads(int32_t Hq, int32_t Hkv, int32_t q_len, int32_t kv_dtype) {
  const int32_t per_head = hpa_default_num_ctas_mma(Hq, Hkv, q_len, kv_dtype);
  if (per_head <= 0) return per_head;
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    cuda_fail(e);
    return -1;
  }
  if (hpa::attn_ctas_per_sm(kv_dtype, q_len, &per_sm) != 0 || per_sm < 1) return -1;
  // one CTA per (partition, group of 16 query rows), each walking every KV head
  const int groups = ((Hq / Hkv) * q_len + hpa::MAX_ROWS - 1) / hpa::MAX_ROWS;
  const int c = sms * per_sm / groups;
  return c < 1 ? 1 : c;
}

size_t hpa_arrivals_elems(int32_t B, int32_t Hq, int32_t Hkv, int32_t q_len) {
  if (B < 1 || B > kMaxB || Hkv < 1 || Hkv > 65535 || Hq < Hkv || Hq % Hkv || q_len < 1)
    return 0;
  const int64_t groups = (int64_t(Hq / Hkv) * q_len + hpa::MAX_ROWS - 1) / hpa::MAX_ROWS;
  return static_cast<size_t>(B) * Hkv * groups;
}

int hpa_decode_attn_fused(const void *q_dev, const void *k_pool_dev, const void *v_pool_dev,
                          int32_t kv_dtype, const float *k_scale_dev, const float *v_scale_dev,
                          int64_t num_pages, const int32_t *page_indptr_dev,
                          const int32_t *page_indices_dev, int32_t page_size, int32_t B,
                          int32_t q_len, int32_t Hq, int32_t Hkv, int32_t d, float sm_scale,
                          void *taskmap_dev, int32_t num_ctas, float *partial_o_dev,
                          float *partial_lse_dev, void *out_dev, float *out_lse_dev,
                          int32_t *arrivals_dev, hpa_stream_t stream) {
  if (!out_dev || !arrivals_dev) return HPA_ERR_INVALID;
  if (!aligned(out_dev, 8) || !aligned(arrivals_dev, 4)) return HPA_ERR_ALIGN;
  return decode_attn_impl(q_dev, k_pool_dev, v_pool_dev, kv_dtype, k_scale_dev, v_scale_dev,
                          num_pages, page_indptr_dev, page_indices_dev, page_size, B, q_len, Hq,
                          Hkv, d, sm_scale, taskmap_dev, num_ctas, partial_o_dev,
                          partial_lse_dev, nullptr, out_dev, out_lse_dev, arrivals_dev, stream);
}

int hpa_combine(const float *partial_o_dev, const float *partial_lse_dev, void *taskmap_dev,
                int32_t B, int32_t num_ctas, int32_t q_len, int32_t Hq, int32_t d,
                void *out_dev, float *out_lse_dev, hpa_stream_t stream) {
  if (!partial_o_dev || !partial_lse_dev || !taskmap_dev || !out_dev) return HPA_ERR_INVALID;
  if (B < 1 || B > kMaxB || num_ctas < 1 || num_ctas > kMaxC || q_len < 1 || Hq < 1)
    return HPA_ERR_INVALID;
  if (d != hpa::HEAD_DIM) return HPA_ERR_UNSUPPORTED;
  if (int64_t(B) * q_len * Hq > INT_MAX) return HPA_ERR_UNSUPPORTED;  // one block per row
  if (!aligned(partial_o_dev, 16) || !aligned(out_dev, 8) || !aligned(taskmap_dev, 16))
    return HPA_ERR_ALIGN;
  cudaError_t e = hpa::launch_combine(partial_o_dev, partial_lse_dev,
                                      static_cast<int32_t *>(taskmap_dev), B, num_ctas, q_len,
                                      Hq, static_cast<__nv_bfloat16 *>(out_dev), out_lse_dev,
                                      reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? HPA_OK : cuda_fail(e);
}

int hpa_selftest_wait_timeout(int32_t *status_dev, int64_t limit_ns, hpa_stream_t stream) {
  if (!status_dev) return HPA_ERR_INVALID;
  if (limit_ns < 1000 || limit_ns > 5000000000ll) return HPA_ERR_INVALID;
  if (!aligned(status_dev, 4)) return HPA_ERR_ALIGN;
  cudaError_t e = hpa::launch_selftest_wait(status_dev, limit_ns,
                                            reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? HPA_OK : cuda_fail(e);
}

int hpa_store_kv(const void *k_new_dev, const void *v_new_dev, const int32_t *seq_lens_dev,
                 const int32_t *page_indptr_dev, const int32_t *page_indices_dev,
                 int64_t num_pages, int32_t page_size, const float *cos_sin_dev, int32_t max_pos,
                 const float *norm_w_dev, float eps, int32_t use_hadamard, int32_t kv_dtype,
                 const float *k_scale_dev, const float *v_scale_dev, void *k_pool_dev,
                 void *v_pool_dev, int32_t B, int32_t q_len, int32_t Hkv, int32_t d,
                 int32_t *status_dev, hpa_stream_t stream) {
  if (!k_new_dev || !v_new_dev || !seq_lens_dev || !page_indptr_dev || !page_indices_dev ||
      !cos_sin_dev || !norm_w_dev || !k_pool_dev || !v_pool_dev)
    return HPA_ERR_INVALID;
  if (kv_dtype != HPA_KV_BF16 && kv_dtype != HPA_KV_E4M3) return HPA_ERR_INVALID;
  if (kv_dtype == HPA_KV_E4M3 && (!k_scale_dev || !v_scale_dev)) return HPA_ERR_INVALID;
  if (B < 1 || B > kMaxB || q_len < 1 || Hkv < 1 || Hkv > 65535 || num_pages < 1 ||
      max_pos < 1 || !(eps >= 0.f) || !std::isfinite(eps))
    return HPA_ERR_INVALID;
  if (d != hpa::HEAD_DIM || page_size != hpa::PAGE) return HPA_ERR_UNSUPPORTED;
  if (int64_t(B) * q_len * Hkv > (int64_t(1) << 34)) return HPA_ERR_UNSUPPORTED;
  if (!aligned(k_new_dev, 16) || !aligned(v_new_dev, 16) || !aligned(cos_sin_dev, 16) ||
      !aligned(norm_w_dev, 16) || !aligned(k_pool_dev, 16) || !aligned(v_pool_dev, 16) ||
      (status_dev && !aligned(status_dev, 4)))
    return HPA_ERR_ALIGN;
  hpa::StoreKvParams p;
  p.k_new = static_cast<const __nv_bfloat16 *>(k_new_dev);
  p.v_new = static_cast<const __nv_bfloat16 *>(v_new_dev);
  p.seq_lens = seq_lens_dev;
  p.page_indptr = page_indptr_dev;
  p.page_indices = page_indices_dev;
  p.num_pages = num_pages;
  p.cos_sin = cos_sin_dev;
  p.max_pos = max_pos;
  p.norm_w = norm_w_dev;
  p.eps = eps;
  p.use_hadamard = use_hadamard != 0;
  p.kv_dtype = kv_dtype;
  p.k_scale = k_scale_dev;
  p.v_scale = v_scale_dev;
  p.k_pool = k_pool_dev;
  p.v_pool = v_pool_dev;
  p.B = B;
  p.q_len = q_len;
  p.Hkv = Hkv;
  p.status = status_dev;
  cudaError_t e = hpa::launch_store_kv(p, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? HPA_OK : cuda_fail(e);
}

const char *hpa_error_string(int code) {
  switch (code) {
    case HPA_OK: return "ok";
    case HPA_ERR_INVALID: return "invalid argument";
    case HPA_ERR_UNSUPPORTED: return "unsupported shape";
    case HPA_ERR_WORKSPACE: return "task map buffer too small";
    case HPA_ERR_ALIGN: return "misaligned pointer";
    case HPA_ERR_CUDA: return "CUDA runtime error";
    case HPA_ERR_NOALLOC_CAPACITY: return "problem exceeds the fixed no-alloc scratch array";
    default: return "unknown error";
  }
}

int hpa_last_cuda_error(void) { return hpa::last_cuda_error(); }

}  // extern "C"
