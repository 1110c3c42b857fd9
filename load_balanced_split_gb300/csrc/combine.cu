// Combine: merges the split-KV partial results of every request by
// log-sum-exp ("Hy3 Preview AI Infra 推理优化精读笔记", §3.1 方案 step 5;
// "腾讯混元AI Infra进化：HPC-Ops推理核心算子全面升级", §二.1 Combine Kernel).
//
// Per (request r, query token j, head g), over r's segments s:
//   M = max lse_s, w_s = exp(lse_s - M), out = sum w_s o_s / sum w_s,
//   out_lse = M + ln sum w_s.
// Lane i owns head dims [4i, 4i+4).  Two kernels, chosen by the number of items:
// - many items (the usual batch): one warp per item, 8 per block.  One pass over the
//   segments, four at a time with their loads in flight together, keeps a running
//   maximum M and rescales the sums by exp(M_old - M_new) when it grows; most
//   requests have one to three segments, so most warps make one round trip.
// - few items (a batch of one or a few long requests, each split over many
//   partitions): one 128-thread block per item; the four warps take every fourth
//   segment with several loads in flight, so a request split over many partitions
//   costs a few round trips, not one per segment.
// A task map whose status word is non-zero makes every output NaN, and so does a
// request whose segment range in the map is out of bounds (reported as
// HPA_STATUS_BAD_MAP).
#include <math_constants.h>

#include "hpa_internal.cuh"

namespace hpa {
namespace {

constexpr int kItemsPerBlock = 8;  // warp-per-item kernel
constexpr int kUnroll = 4;         // its segments in flight per round
constexpr int kBlockWarps = 4;     // block-per-item kernel
constexpr int kBlockUnroll = 4;

// Request r's segment range [s0, s1) from the task map, checked before any partial is
// read through it: false for a map with a non-zero status word, built for another
// shape, or whose range for r is out of bounds (then reported as HPA_STATUS_BAD_MAP
// by the thread with `report` set).
__device__ __forceinline__ bool segment_range(int32_t *tm, int B, int C, int r, bool report,
                                              int &s0, int &s1) {
  s0 = s1 = 0;
  if (!(tm[TM_STATUS] == 0 && tm[TM_B] == B && tm[TM_C] == C)) return false;
  const TaskMapLayout lay = TaskMapLayout::make(B, C);
  s0 = tm[lay.seg_off + r];
  s1 = tm[lay.seg_off + r + 1];
  const int S = tm[TM_S];
  const bool good = s0 >= 0 && s0 < s1 && s1 <= S && S <= B + C - 1;
  if (!good && report) status_or(tm, HPA_STATUS_BAD_MAP);
  return good;
}

// The NaN output of one (request, token, head) item: lane i writes dims [4i, 4i+4).
__device__ __forceinline__ void write_nan(__nv_bfloat16 *out, float *out_lse, int64_t item,
                                          int lane) {
  const float nan = CUDART_NAN_F;
  const __nv_bfloat162 n2 = __floats2bfloat162_rn(nan, nan);
  uint2 pk;
  pk.x = pk.y = *reinterpret_cast<const uint32_t *>(&n2);
  reinterpret_cast<uint2 *>(out + item * HEAD_DIM)[lane] = pk;
  if (out_lse != nullptr && lane == 0) out_lse[item] = nan;
}

__global__ void __launch_bounds__(kItemsPerBlock * 32)
    combine_warp_kernel(const float *__restrict__ po, const float *__restrict__ plse,
                        int32_t *__restrict__ tm, int B, int C, int q_len, int Hq,
                        __nv_bfloat16 *__restrict__ out, float *__restrict__ out_lse) {
  pdl_wait();  // partials come from the attention kernel just before
  const int lane = threadIdx.x & 31;
  const int64_t per_req = static_cast<int64_t>(q_len) * Hq;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * kItemsPerBlock + (threadIdx.x >> 5);
  if (item >= static_cast<int64_t>(B) * per_req) return;
  const int r = static_cast<int>(item / per_req);
  const int64_t jg = item - r * per_req;

  int s0, s1;
  if (!segment_range(tm, B, C, r, lane == 0, s0, s1)) {
    write_nan(out, out_lse, item, lane);
    return;
  }

  float M = -CUDART_INF_F, W = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = s0; s < s1; s += kUnroll) {
    float l[kUnroll];
    float4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int ss = s + u;
      l[u] = -CUDART_INF_F;
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ss < s1) {
        l[u] = plse[ss * per_req + jg];
        v[u] = reinterpret_cast<const float4 *>(po + (ss * per_req + jg) * HEAD_DIM)[lane];
      }
    }
    float mc = l[0];
#pragma unroll
    for (int u = 1; u < kUnroll; ++u) mc = fmaxf(mc, l[u]);
    const float mn = fmaxf(M, mc);
    if (mn == -CUDART_INF_F) continue;  // no visible key in any segment so far
    const float sc = expf(M - mn);      // 0 while M is -inf
    acc.x *= sc, acc.y *= sc, acc.z *= sc, acc.w *= sc;
    W *= sc;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const float wt = expf(l[u] - mn);  // 0 for a missing or empty segment
      acc.x += wt * v[u].x;
      acc.y += wt * v[u].y;
      acc.z += wt * v[u].z;
      acc.w += wt * v[u].w;
      W += wt;
    }
    M = mn;
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 pk;
  pk.x = *reinterpret_cast<const uint32_t *>(&lo);
  pk.y = *reinterpret_cast<const uint32_t *>(&hi);
  reinterpret_cast<uint2 *>(out + item * HEAD_DIM)[lane] = pk;
  if (out_lse != nullptr && lane == 0) out_lse[item] = W > 0.f ? M + logf(W) : -CUDART_INF_F;
}

__global__ void __launch_bounds__(kBlockWarps * 32)
    combine_block_kernel(const float *__restrict__ po, const float *__restrict__ plse,
                         int32_t *__restrict__ tm, int B, int C, int q_len, int Hq,
                         __nv_bfloat16 *__restrict__ out, float *__restrict__ out_lse) {
  pdl_wait();  // partials come from the attention kernel just before
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t item = blockIdx.x;  // (r * q_len + j) * Hq + g
  const int64_t per_req = static_cast<int64_t>(q_len) * Hq;
  const int r = static_cast<int>(item / per_req);
  const int64_t jg = item % per_req;
  __shared__ float s_max[kBlockWarps], s_w[kBlockWarps];
  __shared__ float4 s_acc[kBlockWarps][32];

  int s0, s1;
  if (!segment_range(tm, B, C, r, threadIdx.x == 0, s0, s1)) {
    if (w == 0) write_nan(out, out_lse, item, lane);
    return;
  }

  float m = -CUDART_INF_F;
  for (int s = s0 + threadIdx.x; s < s1; s += kBlockWarps * 32) m = fmaxf(m, plse[s * per_req + jg]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) s_max[w] = m;
  __syncthreads();
  float M = s_max[0];
#pragma unroll
  for (int x = 1; x < kBlockWarps; ++x) M = fmaxf(M, s_max[x]);
  const float Mb = M == -CUDART_INF_F ? 0.f : M;

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float W = 0.f;
  for (int s = s0 + w; s < s1; s += kBlockWarps * kBlockUnroll) {
    float l[kBlockUnroll];
    float4 v[kBlockUnroll];
#pragma unroll
    for (int u = 0; u < kBlockUnroll; ++u) {
      const int ss = s + u * kBlockWarps;
      if (ss < s1) {
        l[u] = plse[ss * per_req + jg];
        v[u] = reinterpret_cast<const float4 *>(po + (ss * per_req + jg) * HEAD_DIM)[lane];
      }
    }
#pragma unroll
    for (int u = 0; u < kBlockUnroll; ++u) {
      if (s + u * kBlockWarps < s1) {
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
  for (int x = 0; x < kBlockWarps; ++x) {
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
  // More than kUnroll segments per request on average (S <= B + C - 1): the
  // block-per-item kernel, whose four warps share an item's segments (a single
  // 192K-token request over 38 partitions: 8.4 against 10.8 us for a warp per item).
  const bool per_block = static_cast<int64_t>(B) + C - 1 > static_cast<int64_t>(kUnroll) * B;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(per_block ? items
                                                     : (items + kItemsPerBlock - 1) / kItemsPerBlock));
  cfg.blockDim = dim3((per_block ? kBlockWarps : kItemsPerBlock) * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, per_block ? combine_block_kernel : combine_warp_kernel, po,
                            static_cast<const float *>(plse), tm, B, C, q_len, Hq, out, out_lse);
}

}  // namespace hpa
