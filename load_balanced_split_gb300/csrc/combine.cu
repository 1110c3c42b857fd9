// Combine: merges the split-KV partial results of every request by
// log-sum-exp ("Hy3 Preview AI Infra 推理优化精读笔记", §3.1 方案 step 5;
// "腾讯混元AI Infra进化：HPC-Ops推理核心算子全面升级", §二.1 Combine Kernel).
//
// One 128-thread block per (request r, query token j, head g).  Over r's
// segments s:
//   M = max lse_s, w_s = exp(lse_s - M), out = sum w_s o_s / sum w_s,
//   out_lse = M + ln sum w_s.
// The four warps take every fourth segment (lane i owns head dims [4i, 4i+4))
// with several loads in flight per warp, so a request split over many
// partitions costs a few round trips, not one per segment.  A task map whose
// status word is non-zero makes every output NaN, and so does a request whose
// segment range in the map is out of bounds (reported as HPA_STATUS_BAD_MAP).
#include <math_constants.h>

#include "hpa_internal.cuh"

namespace hpa {
namespace {

constexpr int kWarps = 4;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kWarps * 32)
    combine_kernel(const float *__restrict__ po, const float *__restrict__ plse,
                   int32_t *__restrict__ tm, int B, int C, int q_len, int Hq,
                   __nv_bfloat16 *__restrict__ out, float *__restrict__ out_lse) {
  pdl_wait();  // partials come from the attention kernel just before
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t item = blockIdx.x;  // (r * q_len + j) * Hq + g
  const int64_t per_req = static_cast<int64_t>(q_len) * Hq;
  const int r = static_cast<int>(item / per_req);
  const int64_t jg = item % per_req;
  __shared__ float s_max[kWarps], s_w[kWarps];
  __shared__ float4 s_acc[kWarps][32];

  const TaskMapLayout lay = TaskMapLayout::make(B, C);
  int s0 = 0, s1 = 0;
  bool good = tm[TM_STATUS] == 0 && tm[TM_B] == B && tm[TM_C] == C;
  if (good) {
    // r's segment range, checked before any partial is read through it
    s0 = tm[lay.seg_off + r];
    s1 = tm[lay.seg_off + r + 1];
    const int S = tm[TM_S];
    good = s0 >= 0 && s0 < s1 && s1 <= S && S <= B + C - 1;
    if (!good && threadIdx.x == 0) status_or(tm, HPA_STATUS_BAD_MAP);
  }
  if (!good) {
    if (w == 0) {
      const float nan = CUDART_NAN_F;
      const __nv_bfloat162 n2 = __floats2bfloat162_rn(nan, nan);
      uint2 pk;
      pk.x = pk.y = *reinterpret_cast<const uint32_t *>(&n2);
      reinterpret_cast<uint2 *>(out + item * HEAD_DIM)[lane] = pk;
      if (out_lse != nullptr && lane == 0) out_lse[item] = nan;
    }
    return;
  }

  float m = -CUDART_INF_F;
  for (int s = s0 + threadIdx.x; s < s1; s += kWarps * 32) m = fmaxf(m, plse[s * per_req + jg]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) s_max[w] = m;
  __syncthreads();
  float M = s_max[0];
#pragma unroll
  for (int x = 1; x < kWarps; ++x) M = fmaxf(M, s_max[x]);
  const float Mb = M == -CUDART_INF_F ? 0.f : M;

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float W = 0.f;
  for (int s = s0 + w; s < s1; s += kWarps * kUnroll) {
    float l[kUnroll];
    float4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int ss = s + u * kWarps;
      if (ss < s1) {
        l[u] = plse[ss * per_req + jg];
        v[u] = reinterpret_cast<const float4 *>(po + (ss * per_req + jg) * HEAD_DIM)[lane];
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (s + u * kWarps < s1) {
        const float wt = expf(l[u] - Mb);
        acc.x += wt * v[u].x;
        acc.y += wt * v[u].y;
        acc.z += wt * v[u].z;
        acc.w += wt * v[u].w;
        W += wt;
      }
    }
  }
  s_acc[w][lane] = acc;
  if (lane == 0) s_w[w] = W;
  __syncthreads();
  if (w != 0) return;
  float Wt = 0.f;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int x = 0; x < kWarps; ++x) {
    const float4 t = s_acc[x][lane];
    a.x += t.x;
    a.y += t.y;
    a.z += t.z;
    a.w += t.w;
    Wt += s_w[x];
  }
  const float inv = Wt > 0.f ? 1.f / Wt : 0.f;
  const __nv_bfloat162 lo = __floats2bfloat162_rn(a.x * inv, a.y * inv);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(a.z * inv, a.w * inv);
  uint2 pk;
  pk.x = *reinterpret_cast<const uint32_t *>(&lo);
  pk.y = *reinterpret_cast<const uint32_t *>(&hi);
  reinterpret_cast<uint2 *>(out + item * HEAD_DIM)[lane] = pk;
  if (out_lse != nullptr && lane == 0) out_lse[item] = Wt > 0.f ? Mb + logf(Wt) : -CUDART_INF_F;
}

}  // namespace

cudaError_t launch_combine(const float *po, const float *plse, int32_t *tm, int B, int C,
                           int q_len, int Hq, __nv_bfloat16 *out, float *out_lse,
                           cudaStream_t s) {
  const int64_t items = static_cast<int64_t>(B) * q_len * Hq;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(items));
  cfg.blockDim = dim3(kWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, po, static_cast<const float *>(plse), tm, B,
                            C, q_len, Hq, out, out_lse);
}

}  // namespace hpa
