// Fused KV-cache writer: RoPE + RMSNorm + Hadamard + quantisation + paged store,
// one pass ("Hy3 Preview AI Infra 推理优化精读笔记", §4.1 "Rope + Norm + Hadamard +
// Quant + Store KV": the element-wise chain after the QKV projection, fused so
// the new keys and values go from registers straight into the low-bit cache).
//
// One warp per (request r, new token j), four KV heads at a time (8 lanes per
// head, 16 dims per lane).  For the key: rotate-half RoPE with the caller's
// cos/sin table, RMSNorm over the 128 dims, optional orthonormal Walsh-Hadamard
// transform, then E4M3 codes of x / scale (round to nearest even, saturating)
// or bf16.  The value is only converted.  Token j of request r is written at
// position L_r - q_len + j.
#include "hpa_internal.cuh"

namespace hpa {
namespace {

constexpr int kWarps = 8;
constexpr uint32_t kFull = 0xffffffffu;

// Lane layout: a warp handles 4 KV heads at a time, 8 lanes per head; lane k of
// a head's group holds dims [8k, 8k + 8) and [64 + 8k, 64 + 8k + 8) -- so each
// RoPE pair (i, i + 64) is inside one lane, and of the 7 butterfly stages of the
// 128-point Walsh-Hadamard transform, 4 (dim bits 0-2 and 6) are in registers
// and 3 (bits 3-5: lane bits 0-2) cross lanes.
constexpr int kLanesPerHead = 8;
constexpr int kHeadsPerPass = 32 / kLanesPerHead;

constexpr int kPasses = 2;  // passes of 4 heads whose rows are loaded together

__device__ __forceinline__ void unpack16(const uint4 (&raw)[2], float (&x)[16]) {
  const uint4 a = raw[0], b = raw[1];
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

// x[0..7] -> dims 8k.., x[8..15] -> dims 64 + 8k.. of pool row `row`.
__device__ __forceinline__ void store16(void *pool, int kv_dtype, int64_t row, int k,
                                        const float (&x)[16], float inv_scale) {
  if (kv_dtype == HPA_KV_BF16) {
    __nv_bfloat16 *base = static_cast<__nv_bfloat16 *>(pool) + row * HEAD_DIM;
    uint4 a, b;
    a.x = pack_bf16(x[0], x[1]), a.y = pack_bf16(x[2], x[3]);
    a.z = pack_bf16(x[4], x[5]), a.w = pack_bf16(x[6], x[7]);
    b.x = pack_bf16(x[8], x[9]), b.y = pack_bf16(x[10], x[11]);
    b.z = pack_bf16(x[12], x[13]), b.w = pack_bf16(x[14], x[15]);
    reinterpret_cast<uint4 *>(base + 8 * k)[0] = a;
    reinterpret_cast<uint4 *>(base + 64 + 8 * k)[0] = b;
  } else {
    uint8_t *base = static_cast<uint8_t *>(pool) + row * HEAD_DIM;
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = f32x2_to_e4m3x2(x[4 * i] * inv_scale, x[4 * i + 1] * inv_scale);
      const uint32_t hi = f32x2_to_e4m3x2(x[4 * i + 2] * inv_scale, x[4 * i + 3] * inv_scale);
      q[i] = lo | (hi << 16);
    }
    reinterpret_cast<uint2 *>(base + 8 * k)[0] = make_uint2(q[0], q[1]);
    reinterpret_cast<uint2 *>(base + 64 + 8 * k)[0] = make_uint2(q[2], q[3]);
  }
}

// RoPE + RMSNorm + (Hadamard) of one key row, 16 dims in this lane (see above).
__device__ __forceinline__ void key_transform(float (&y)[16], const float (&c)[8],
                                              const float (&sn)[8], const float (&w)[16],
                                              float eps, int use_hadamard) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {  // rotate-half RoPE: (y_i, y_{i+64}) turned by angle i
    const float lo = y[i], hi = y[8 + i];
    y[i] = lo * c[i] - hi * sn[i];
    y[8 + i] = hi * c[i] + lo * sn[i];
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) ss += y[i] * y[i];
  ss += __shfl_xor_sync(kFull, ss, 1);
  ss += __shfl_xor_sync(kFull, ss, 2);
  ss += __shfl_xor_sync(kFull, ss, 4);
  const float inv = rsqrtf(ss / HEAD_DIM + eps);
#pragma unroll
  for (int i = 0; i < 16; ++i) y[i] *= inv * w[i];
  if (!use_hadamard) return;
  // orthonormal Walsh-Hadamard transform, Sylvester order: a butterfly
  // (a, b) -> (a + b, a - b) over every dim bit; in-register bits 0-2 and 6
#pragma unroll
  for (int st = 1; st < 16; st <<= 1) {  // register index bit: 1,2,4 -> dim bits 0-2; 8 -> bit 6
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (!(i & st)) {
        const float a = y[i], b = y[i | st];
        y[i] = a + b;
        y[i | st] = a - b;
      }
  }
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 1; m < kLanesPerHead; m <<= 1) {  // dim bits 3-5: partner lane ^ m
    const bool up = lane & m;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float p = __shfl_xor_sync(kFull, y[i], m);
      y[i] = up ? p - y[i] : y[i] + p;
    }
  }
  const float n = 0.08838834764831845f;  // 1 / sqrt(128)
#pragma unroll
  for (int i = 0; i < 16; ++i) y[i] *= n;
}

// One warp per new token (r, j): the position, page and RoPE row are looked up
// once and shared by the token's KV heads, four heads per pass.
__global__ void __launch_bounds__(kWarps * 32, 2)
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
  const int k = lane % kLanesPerHead, hp = lane / kLanesPerHead;
  const int64_t rj = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (rj >= static_cast<int64_t>(B) * q_len) return;
  const int r = static_cast<int>(rj / q_len), j = static_cast<int>(rj % q_len);
  const int64_t src0 = rj * Hkv * HEAD_DIM;
  // raw bf16 rows of this lane's heads, kPasses x 4 heads per block, loaded before
  // they are needed so a token's K and V (4 KB for 8 heads) is in flight at once
  uint4 kraw[kPasses][2], vraw[kPasses][2];
  auto load_block = [&](int hb) {
#pragma unroll
    for (int ps = 0; ps < kPasses; ++ps) {
      const int h = hb + ps * kHeadsPerPass + hp;
      if (h < Hkv) {
        const __nv_bfloat16 *kr = k_new + src0 + static_cast<int64_t>(h) * HEAD_DIM;
        const __nv_bfloat16 *vr = v_new + src0 + static_cast<int64_t>(h) * HEAD_DIM;
        kraw[ps][0] = reinterpret_cast<const uint4 *>(kr + 8 * k)[0];
        kraw[ps][1] = reinterpret_cast<const uint4 *>(kr + 64 + 8 * k)[0];
        vraw[ps][0] = reinterpret_cast<const uint4 *>(vr + 8 * k)[0];
        vraw[ps][1] = reinterpret_cast<const uint4 *>(vr + 64 + 8 * k)[0];
      }
    }
  };
  load_block(0);  // independent of the page lookup below

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
  float c[8], sn[8], w[16];
  {
    const float4 *cs = reinterpret_cast<const float4 *>(cos_sin + static_cast<int64_t>(pos) * HEAD_DIM);
    const float4 c0 = cs[2 * k], c1 = cs[2 * k + 1];             // cos of dims 8k..8k+7
    const float4 s0 = cs[16 + 2 * k], s1 = cs[16 + 2 * k + 1];   // sin of the same
    const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = cc[i], sn[i] = ss[i];
    const float4 *wv = reinterpret_cast<const float4 *>(norm_w);
    const float4 w0 = wv[2 * k], w1 = wv[2 * k + 1], w2 = wv[16 + 2 * k], w3 = wv[16 + 2 * k + 1];
    const float ww[16] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w,
                          w2.x, w2.y, w2.z, w2.w, w3.x, w3.y, w3.z, w3.w};
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = ww[i];
  }
  const bool e4m3 = kv_dtype == HPA_KV_E4M3;
  for (int hb = 0; hb < Hkv; hb += kPasses * kHeadsPerPass) {
    if (hb > 0) load_block(hb);
#pragma unroll
  for (int ps = 0; ps < kPasses; ++ps) {
    const int h = hb + ps * kHeadsPerPass + hp;
    const bool active = h < Hkv;  // lanes of a missing head still take the shuffles
    float y[16], x[16];
    if (active) {
      unpack16(kraw[ps], y);
      unpack16(vraw[ps], x);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) y[i] = x[i] = 0.f;
    }
    key_transform(y, c, sn, w, eps, use_hadamard);
    if (active) {
      const int64_t row = (static_cast<int64_t>(page) * Hkv + h) * PAGE + pos % PAGE;
      store16(k_pool, kv_dtype, row, k, y, e4m3 ? 1.f / k_scale[h] : 1.f);
      store16(v_pool, kv_dtype, row, k, x, e4m3 ? 1.f / v_scale[h] : 1.f);  // value: converted only
    }
  }
  }
}

}  // namespace

cudaError_t launch_store_kv(const StoreKvParams &p, cudaStream_t s) {
  const int64_t items = static_cast<int64_t>(p.B) * p.q_len;  // one warp per new token
  const unsigned blocks = static_cast<unsigned>((items + kWarps - 1) / kWarps);
  store_kv_kernel<<<blocks, kWarps * 32, 0, s>>>(
      p.k_new, p.v_new, p.seq_lens, p.page_indptr, p.page_indices, p.num_pages, p.cos_sin,
      p.max_pos, p.norm_w, p.eps, p.use_hadamard, p.kv_dtype, p.k_scale, p.v_scale, p.k_pool,
      p.v_pool, p.B, p.q_len, p.Hkv, p.status);
  return cudaGetLastError();
}

}  // namespace hpa
