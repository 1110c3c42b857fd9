// Combine: merges the split-KV partial results of every request by
// log-sum-exp ("Hy3 Preview AI Infra 推理优化精读笔记", §3.1 方案 step 5;
// "腾讯混元AI Infra进化：HPC-Ops推理核心算子全面升级", §二.1 Combine Kernel).
//
// One warp per (request r, query token j, head g); lane i owns head dims
// [4i, 4i+4).  Over r's segments s:
//   M = max lse_s, w_s = exp(lse_s - M), out = sum w_s o_s / sum w_s,
//   out_lse = M + ln sum w_s.
// A task map whose status word is non-zero makes every output NaN.
#include <math_constants.h>

#include "hpa_internal.cuh"

namespace hpa {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32)
    combine_kernel(const float *__restrict__ po, const float *__restrict__ plse,
                   const int32_t *__restrict__ tm, int B, int C, int q_len, int Hq,
                   __nv_bfloat16 *__restrict__ out, float *__restrict__ out_lse) {
  const int lane = threadIdx.x & 31;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t n_items = static_cast<int64_t>(B) * q_len * Hq;
  if (item >= n_items) return;
  const int r = static_cast<int>(item / (static_cast<int64_t>(q_len) * Hq));
  const int jg = static_cast<int>(item % (static_cast<int64_t>(q_len) * Hq));  // j * Hq + g
  const TaskMapLayout lay = TaskMapLayout::make(B, C);
  const bool bad = tm[TM_STATUS] != 0 || tm[TM_B] != B || tm[TM_C] != C;

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float lse;
  if (bad) {
    acc = make_float4(CUDART_NAN_F, CUDART_NAN_F, CUDART_NAN_F, CUDART_NAN_F);
    lse = CUDART_NAN_F;
  } else {
    const int s0 = tm[lay.seg_off + r], s1 = tm[lay.seg_off + r + 1];
    const int64_t stride = static_cast<int64_t>(q_len) * Hq;  // per segment
    float M = -CUDART_INF_F;
    for (int s = s0 + lane; s < s1; s += 32) M = fmaxf(M, plse[s * stride + jg]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float Mb = M == -CUDART_INF_F ? 0.f : M;
    float W = 0.f;
    for (int s = s0; s < s1; ++s) {
      const float w = expf(plse[s * stride + jg] - Mb);
      const float4 v =
          reinterpret_cast<const float4 *>(po + (s * stride + jg) * HEAD_DIM)[lane];
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
      W += w;
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
    lse = W > 0.f ? Mb + logf(W) : -CUDART_INF_F;
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t *>(&lo);
  pk.y = *reinterpret_cast<uint32_t *>(&hi);
  reinterpret_cast<uint2 *>(out + item * HEAD_DIM)[lane] = pk;
  if (out_lse != nullptr && lane == 0) out_lse[item] = lse;
}

}  // namespace

cudaError_t launch_combine(const float *po, const float *plse, int32_t *tm, int B, int C,
                           int q_len, int Hq, __nv_bfloat16 *out, float *out_lse,
                           cudaStream_t s) {
  const int64_t items = static_cast<int64_t>(B) * q_len * Hq;
  const int64_t blocks = (items + kWarps - 1) / kWarps;
  combine_kernel<<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(po, plse, tm, B, C,
                                                                       q_len, Hq, out, out_lse);
  return cudaGetLastError();
}

}  // namespace hpa
