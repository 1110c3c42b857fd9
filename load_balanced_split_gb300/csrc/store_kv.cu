// Fused KV-cache writer: RoPE + RMSNorm + Hadamard + quantisation + paged store,
// one pass ("Hy3 Preview AI Infra 推理优化精读笔记", §4.1 "Rope + Norm + Hadamard +
// Quant + Store KV": the element-wise chain after the QKV projection, fused so
// the new keys and values go from registers straight into the low-bit cache).
//
// One warp per (request r, new token j, KV head h); lane i owns head dims
// [4i, 4i + 4).  For the key: rotate-half RoPE with the caller's cos/sin table
// (the partner of dim x is dim x +- 64, held by lane i ^ 16), RMSNorm over the
// 128 dims (warp reduction), optional orthonormal Walsh-Hadamard transform
// (two butterfly stages inside the lane, five across lanes), then E4M3 codes of
// x / scale (round to nearest even, saturating) or bf16.  The value is only
// converted.  Token j of request r is written at position L_r - q_len + j.
#include "hpa_internal.cuh"

namespace hpa {
namespace {

constexpr int kWarps = 8;
constexpr uint32_t kFull = 0xffffffffu;

__device__ __forceinline__ void store4(void *pool, int kv_dtype, int64_t row, int lane, float4 x,
                                       float inv_scale) {
  if (kv_dtype == HPA_KV_BF16) {
    uint2 pk;
    pk.x = pack_bf16(x.x, x.y);
    pk.y = pack_bf16(x.z, x.w);
    reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(pool) + row * HEAD_DIM)[lane] = pk;
  } else {
    const uint32_t lo = f32x2_to_e4m3x2(x.x * inv_scale, x.y * inv_scale);
    const uint32_t hi = f32x2_to_e4m3x2(x.z * inv_scale, x.w * inv_scale);
    reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(pool) + row * HEAD_DIM)[lane] =
        lo | (hi << 16);
  }
}

__global__ void __launch_bounds__(kWarps * 32)
    store_kv_kernel(const __nv_bfloat16 *__restrict__ k_new,
                    const __nv_bfloat16 *__restrict__ v_new, const int32_t *__restrict__ seq_lens,
                    const int32_t *__restrict__ page_indptr,
                    const int32_t *__restrict__ page_indices, int64_t num_pages,
                    const float *__restrict__ cos_sin, int max_pos,
                    const float *__restrict__ norm_w, float eps, int use_hadamard, int kv_dtype,
                    const float *__restrict__ k_scale, const float *__restrict__ v_scale,
                    void *k_pool, void *v_pool, int B, int q_len, int Hkv,
                    int32_t *__restrict__ status) {
  const int lane = threadIdx.x & 31;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (item >= static_cast<int64_t>(B) * q_len * Hkv) return;
  const int h = static_cast<int>(item % Hkv);
  const int64_t rj = item / Hkv;  // r * q_len + j
  const int r = static_cast<int>(rj / q_len), j = static_cast<int>(rj % q_len);

  const int pos = seq_lens[r] - q_len + j;
  if (pos < 0 || pos >= max_pos) {
    if (lane == 0 && status) atomicOr(reinterpret_cast<int *>(status), HPA_STATUS_BAD_SEQLEN);
    return;
  }
  const int pi = page_indptr[r] + pos / PAGE;
  const int page = pi < page_indptr[r + 1] ? page_indices[pi] : -1;
  if (page < 0 || page >= num_pages) {
    if (lane == 0 && status) atomicOr(reinterpret_cast<int *>(status), HPA_STATUS_BAD_PAGE);
    return;
  }
  const int64_t row = (static_cast<int64_t>(page) * Hkv + h) * PAGE + pos % PAGE;

  // ---- key: RoPE (rotate half)
  const int64_t src = (rj * Hkv + h) * HEAD_DIM;
  const uint2 kr = reinterpret_cast<const uint2 *>(k_new + src)[lane];
  float x[4];
  {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kr.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kr.y));
    x[0] = a.x, x[1] = a.y, x[2] = b.x, x[3] = b.y;
  }
  const bool upper = lane >= 16;  // dims 64..127: the second half of each pair
  const float4 cs_c = reinterpret_cast<const float4 *>(cos_sin + static_cast<int64_t>(pos) * HEAD_DIM)[lane & 15];
  const float4 cs_s =
      reinterpret_cast<const float4 *>(cos_sin + static_cast<int64_t>(pos) * HEAD_DIM + HEAD_DIM / 2)[lane & 15];
  const float c4[4] = {cs_c.x, cs_c.y, cs_c.z, cs_c.w}, s4[4] = {cs_s.x, cs_s.y, cs_s.z, cs_s.w};
  float y[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float partner = __shfl_xor_sync(kFull, x[e], 16);
    y[e] = upper ? x[e] * c4[e] + partner * s4[e] : x[e] * c4[e] - partner * s4[e];
  }
  // ---- RMSNorm over the head dim
  float ss = y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
  const float inv = rsqrtf(ss / HEAD_DIM + eps);
  const float4 w = reinterpret_cast<const float4 *>(norm_w)[lane];
  y[0] *= inv * w.x;
  y[1] *= inv * w.y;
  y[2] *= inv * w.z;
  y[3] *= inv * w.w;
  // ---- orthonormal Walsh-Hadamard transform (Sylvester order) over the 128 dims
  if (use_hadamard) {
    float t0 = y[0] + y[1], t1 = y[0] - y[1], t2 = y[2] + y[3], t3 = y[2] - y[3];  // stride 1
    y[0] = t0 + t2, y[2] = t0 - t2, y[1] = t1 + t3, y[3] = t1 - t3;                // stride 2
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {  // strides 4 .. 64: partner lane i ^ m
      const bool hi = lane & m;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = __shfl_xor_sync(kFull, y[e], m);
        y[e] = hi ? p - y[e] : y[e] + p;
      }
    }
    const float n = 0.08838834764831845f;  // 1 / sqrt(128)
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] *= n;
  }
  const bool e4m3 = kv_dtype == HPA_KV_E4M3;
  store4(k_pool, kv_dtype, row, lane, make_float4(y[0], y[1], y[2], y[3]),
         e4m3 ? 1.f / k_scale[h] : 1.f);

  // ---- value: converted only
  const uint2 vr = reinterpret_cast<const uint2 *>(v_new + src)[lane];
  const float2 va = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&vr.x));
  const float2 vb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&vr.y));
  store4(v_pool, kv_dtype, row, lane, make_float4(va.x, va.y, vb.x, vb.y),
         e4m3 ? 1.f / v_scale[h] : 1.f);
}

}  // namespace

cudaError_t launch_store_kv(const StoreKvParams &p, cudaStream_t s) {
  const int64_t items = static_cast<int64_t>(p.B) * p.q_len * p.Hkv;
  const unsigned blocks = static_cast<unsigned>((items + kWarps - 1) / kWarps);
  store_kv_kernel<<<blocks, kWarps * 32, 0, s>>>(
      p.k_new, p.v_new, p.seq_lens, p.page_indptr, p.page_indices, p.num_pages, p.cos_sin,
      p.max_pos, p.norm_w, p.eps, p.use_hadamard, p.kv_dtype, p.k_scale, p.v_scale, p.k_pool,
      p.v_pool, p.B, p.q_len, p.Hkv, p.status);
  return cudaGetLastError();
}

}  // namespace hpa
