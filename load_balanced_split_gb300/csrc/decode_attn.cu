// Split-KV GQA decode attention over a paged KV cache, driven by a task map.
//
// "Hy3 Preview AI Infra 推理优化精读笔记", §3.1 方案 steps 4-5: every attention CTA
// takes the tiles the task map gives it and writes split-KV partial results
// for a later combine.  Here one CTA is (partition c, KV head h): it walks the
// segments of partition c and, per segment, reduces the segment's keys for
// the G query heads of h and every new query token (rows = G * q_len <= 16).
//
// GB300 design:
//  * one warp of TMA producer + four consumer warps, 2 CTAs per SM;
//  * a page of one KV head (64 tokens x 128 dims; 16 KB bf16 / 8 KB E4M3 for K
//    and again for V) is one pipeline stage, fetched with 3-D tiled TMA copies
//    in 128-byte-swizzled form so the consumers' shared-memory reads are free
//    of bank conflicts; completion is tracked with mbarriers;
//  * each consumer warp owns 16 of the page's 64 keys: S = Q K^T and O += P V
//    run as m16n8k16 tensor-core MMAs with the query rows as M (16 rows: the
//    8 heads of the group x up to 2 tokens), keys as N / K;
//  * FP32 online softmax in base 2 (scores pre-multiplied by sm_scale*log2 e),
//    per-warp running (m, l, O) merged across the 4 warps at each segment end;
//  * E4M3 pages are widened to f16 in registers (exact), with a consistent
//    permutation of the head dimension between Q and K and of the output
//    columns for V, so every shared-memory read is a 16-byte vector load;
//  * every wait is bounded in time; a CTA that gives up flags the task map's
//    status word, waits for its own copies in flight and returns.
#include <math_constants.h>

#include <type_traits>

#include "hpa_internal.cuh"

namespace hpa {
namespace {

constexpr int kConsumerWarps = 4;
// Segment-end merge buffers (two): one row of 128 partial-output columns per
// query row.  Warps 0 / 1 store into buffers A / B, warps 2 / 3 add into them, and
// the read-out sums A + B: plain shared-memory traffic, no atomics.
//  * bf16: the accumulators hold dim 8 i + n (n-tile i, column n); rows of 136
//    floats keep a warp's float2 fragment stores at 2 lanes per bank at most;
//  * E4M3: a thread holds the 32 contiguous dims [32 qd, 32 qd + 32) of its two
//    rows (the output-column permutation of the 8-bit V path), so it stores them
//    as float4s in dim order; each 32-dim chunk is padded by 4 floats (rows of
//    144) so those stores take the minimum 4 wavefronts, and the read-out loads
//    float4s.
template <int KV>
constexpr int kMergeStrideOf = KV == HPA_KV_E4M3 ? HEAD_DIM + 16 : HEAD_DIM + 8;
__host__ __device__ constexpr int merge_phys(int dd) { return dd + 4 * (dd >> 5); }
// Largest score excess (log2 units) over the running reference max before the
// accumulators are rescaled: P values stay <= 256, well inside bf16/f16 range.
constexpr float kRescaleSlack = 8.f;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr uint32_t kFull = 0xffffffffu;

template <int KV>
struct Cfg;
// Ring depth: bf16 pages stream best with few bytes in flight per CTA (two
// 32 KB stages: fairer sharing of DRAM between the CTAs of one wave, a shorter
// tail); E4M3 consumers do more work per byte and want a deeper ring.
template <>
struct Cfg<HPA_KV_BF16> {
  static constexpr int kKBytes = 16384;  // one page-head of K: 64 x 128 bf16
  static constexpr int kStages = 2;
};
template <>
struct Cfg<HPA_KV_E4M3> {
  static constexpr int kKBytes = 8192;  // 64 x 128 bytes
  static constexpr int kStages = 5;
};

// Per-segment staging written by the producer warp ahead of the consumers: the
// segment's (request, length, key range) and its query rows, in a 2-slot ring.
// Query rows are 256 B padded to 272 B so fragment loads are free of conflicts.
constexpr int kQRowBytes = 272;
constexpr int kQSlotBytes = MAX_ROWS * kQRowBytes;

template <int KV>
struct Smem {
  static constexpr int kStageBytes = 2 * Cfg<KV>::kKBytes;
  static constexpr int kStages = Cfg<KV>::kStages;
  static constexpr int kMergeStride = kMergeStrideOf<KV>;
  static constexpr int kMerge = kStages * kStageBytes;  // float[2][16][kMergeStride]
  static constexpr int kStats = kMerge + 2 * MAX_ROWS * kMergeStride * 4;  // m[4][16], l[4][16]
  static constexpr int kQ = kStats + 2 * kConsumerWarps * MAX_ROWS * 4;  // 2 query slots
  static constexpr int kInfo = kQ + 2 * kQSlotBytes;                      // int4[2][2]
  static constexpr int kBars = kInfo + 4 * 16;  // full[kStages] empty[kStages] qfull[2] qempty[2]
  static constexpr int kFlag = kBars + (2 * kStages + 4) * 8;
  static constexpr int kBytes = kFlag + 16;  // abort flag, last-arriver flag
  static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024 B
};

// Query rows are handled in groups of 16 (one m16 MMA tile): CTA z of a
// (partition, head) pair takes rows [16 z, 16 z + 16) of the G * q_len rows,
// so MTP with more draft tokens (up to 64 rows) reuses the same kernel.
__device__ __forceinline__ int row_base() { return MAX_ROWS * static_cast<int>(blockIdx.z); }
__device__ __forceinline__ int group_rows(const AttnParams &p) {
  return min(MAX_ROWS, p.rows - row_base());
}

struct SegInfo {
  int r, L, klo, khi, pg0, pg1;
};

// Segment s of partition c, checked (a malformed row reads as an empty segment).
__device__ __forceinline__ SegInfo seg_info(const AttnParams &p, int s, int tile, int c,
                                            bool report) {
  const SegRow sr = read_seg_row(p.tm, p.lay, p.B, s, c, tile, report);
  SegInfo f;
  f.r = sr.r;
  f.L = sr.L;
  f.klo = sr.klo;
  f.khi = sr.khi;
  f.pg0 = f.klo / PAGE;
  f.pg1 = (f.khi + PAGE - 1) / PAGE;
  return f;
}

// ----------------------------------------------------------------------------- producer
template <int KV, bool FUSED, bool ALLH>
__device__ void producer(const AttnParams &p, const CUtensorMap *tmk, const CUtensorMap *tmv,
                         uint8_t *smem, int s_begin, int s_end, int tile, int h0) {
  using S = Smem<KV>;
  const int lane = threadIdx.x & 31;
  const uint32_t base = smem_u32(smem);
  const uint32_t full0 = base + S::kBars, empty0 = full0 + 8 * S::kStages;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kFlag);
  uint64_t pol = 0;
  if (lane == 0) {
    pol = l2_policy_evict_first();
    prefetch_tmap(tmk);
    prefetch_tmap(tmv);
  }
  const uint32_t qfull0 = empty0 + 8 * S::kStages, qempty0 = qfull0 + 16;
  int stage = 0;
  uint32_t phase = 0, issued = 0, parity_bits = 0;
  bool ok = true;
  // work items: (segment, KV head), heads innermost; one head per CTA on the
  // per-head grid, all of them with heads_per_cta == Hkv
  const int hpc = ALLH ? p.heads_per_cta : 1, n_items = (s_end - s_begin) * hpc;
  for (int k = 0; k < n_items && ok; ++k) {
    const int s = s_begin + k / hpc, h = h0 + k % hpc;
    const SegInfo f = seg_info(p, s, tile, blockIdx.x, lane == 0 && h == h0);
    // stage the item's segment info and query rows for the consumers
    {
      const int slot = k & 1;
      const uint32_t qphase = (k >> 1) & 1;
      int good = 1;
      if (lane == 0) good = !*abort_flag && mbar_wait_bounded(qempty0 + 8 * slot, qphase ^ 1);
      if (!__shfl_sync(kFull, good, 0)) {
        ok = false;
        break;
      }
      uint8_t *qs = smem + S::kQ + slot * kQSlotBytes;
      const int G = p.G, rb = row_base();
      for (int ch = lane; ch < group_rows(p) * 16; ch += 32) {  // 16-B chunks of 256-B rows
        const int row = ch >> 4, c16 = ch & 15, j = (rb + row) / G, g = (rb + row) % G;
        const int4 v = reinterpret_cast<const int4 *>(
            p.q + ((static_cast<int64_t>(f.r) * p.q_len + j) * p.Hq + h * G + g) * HEAD_DIM)[c16];
        *reinterpret_cast<int4 *>(qs + row * kQRowBytes + c16 * 16) = v;
      }
      if (lane == 0) {
        int4 *info = reinterpret_cast<int4 *>(smem + S::kInfo) + 2 * slot;
        info[0] = make_int4(f.r, f.L, f.klo, f.khi);
        if (FUSED) {  // fused combine: the request's segment range, which must hold s
          const int so = p.tm[p.lay.seg_off + f.r], so1 = p.tm[p.lay.seg_off + f.r + 1];
          const bool good_range = so >= 0 && so <= s && s < so1 && so1 <= p.B + p.C - 1;
          if (!good_range) status_or(p.tm, HPA_STATUS_BAD_MAP);  // no merge for it
          info[1] = make_int4(good_range ? so : 0, good_range ? so1 - so : 0, 0, 0);
        }
      }
      mbar_arrive(qfull0 + 8 * slot);  // every lane publishes its own stores
    }
    const int pstart = p.page_indptr[f.r];
    const int pcount = p.page_indptr[f.r + 1] - pstart;  // pages listed for request r
    const int32_t *pidx = p.page_indices + pstart;
    for (int pb = f.pg0; pb < f.pg1 && ok; pb += 32) {
      const int cnt = min(32, f.pg1 - pb);
      int id = 0;
      if (lane < cnt) {
        id = pb + lane < pcount ? pidx[pb + lane] : -1;
        if (id < 0 || id >= p.num_pages) {  // bad id or too short a page list
          status_or(p.tm, HPA_STATUS_BAD_PAGE);
          id = 0;
        }
      }
      for (int i = 0; i < cnt; ++i) {
        const int pid = __shfl_sync(kFull, id, i);
        int good = 1;
        if (lane == 0) {
          if (*abort_flag || !mbar_wait_bounded(empty0 + 8 * stage, phase ^ 1)) {
            good = 0;
          } else {
            const uint32_t fb = full0 + 8 * stage;
            const uint32_t dst = base + stage * S::kStageBytes;
            const int z = pid * p.Hkv + h;
            mbar_arrive_expect_tx(fb, S::kStageBytes);
            if (KV == HPA_KV_BF16) {
              tma_load_3d(dst, tmk, fb, 0, 0, z, pol);
              tma_load_3d(dst + 8192, tmk, fb, 64, 0, z, pol);
              tma_load_3d(dst + 16384, tmv, fb, 0, 0, z, pol);
              tma_load_3d(dst + 24576, tmv, fb, 64, 0, z, pol);
            } else {
              tma_load_3d(dst, tmk, fb, 0, 0, z, pol);
              tma_load_3d(dst + 8192, tmv, fb, 0, 0, z, pol);
            }
            issued |= 1u << stage;
            parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
          }
        }
        ok = __shfl_sync(kFull, good, 0) != 0;
        if (!ok) break;
        if (++stage == S::kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  }
  if (!ok && lane == 0) {
    status_or(p.tm, HPA_STATUS_TIMEOUT);
    *abort_flag = 1;
    // never leave the CTA with copies still landing in its shared memory
    for (int st = 0; st < S::kStages; ++st)
      if (issued & (1u << st))
        mbar_wait_bounded(full0 + 8 * st, (parity_bits >> st) & 1u, 1000000000ull);
  }
}

// ----------------------------------------------------------------------------- consumer helpers
// Largest |x| of four consecutive bf16 values (8-byte aligned).
__device__ __forceinline__ float absmax4_bf16(const __nv_bfloat16 *x) {
  const uint2 raw = *reinterpret_cast<const uint2 *>(x);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.y));
  return fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(b.x), fabsf(b.y)));
}

// e such that amax * 2^e lies in [2^14, 2^15) (0 for a zero row), clamped so that
// both 2^e and 2^-e are fp32 normals.
__device__ __forceinline__ int f16_row_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  const int ea = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127;  // floor(log2)
  return 14 - min(max(ea, -112), 126);
}

// Zero the V rows (keys >= L) this warp reads from a page that ends past L.
template <int KV>
__device__ __forceinline__ void zero_tail_rows(uint8_t *vtile, int w, int wk, int L, int lane) {
  const int4 z = make_int4(0, 0, 0, 0);
  if (KV == HPA_KV_BF16) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int id = lane + 32 * i, rr = id >> 4, hf = (id >> 3) & 1, ch = id & 7;
      if (wk + rr >= L)
        *reinterpret_cast<int4 *>(vtile + hf * 8192 + (16 * w + rr) * 128 + ch * 16) = z;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int id = lane + 32 * i, rr = id >> 3, ch = id & 7;
      if (wk + rr >= L) *reinterpret_cast<int4 *>(vtile + (16 * w + rr) * 128 + ch * 16) = z;
    }
  }
}

// S[16 rows x 16 keys] = Q K^T for the warp's keys of the page in `kt`.
template <int KV>
__device__ __forceinline__ void qk(float (&s)[2][4], const uint32_t (&qa)[8][4], uint32_t kt,
                                   int w, int lane) {
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
  if (KV == HPA_KV_BF16) {
    const int mi = lane >> 3, key = 16 * w + (mi >> 1) * 8 + (lane & 7);
    const uint32_t row = kt + key * 128;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int chunk = (ks & 3) * 2 + (mi & 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(row + (ks >> 2) * 8192 + ((chunk ^ (lane & 7)) << 4), b0, b1, b2, b3);
      mma_bf16(s[0], qa[ks], b0, b1);
      mma_bf16(s[1], qa[ks], b2, b3);
    }
  } else {
    // thread (r8, qd) reads head dims [32 qd, 32 qd + 32) of its key row and widens
    // them to f16; k-step ks covers dims 32 qd + 4 ks + [0, 4), the same
    // permutation of the head dimension the query fragments use.
    const int r8 = lane >> 2, qd = lane & 3;
    uint32_t u[2][8];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const uint32_t row = kt + (16 * w + 8 * nt + r8) * 128;
      lds128(row + (((2 * qd) ^ r8) << 4), u[nt][0], u[nt][1], u[nt][2], u[nt][3]);
      lds128(row + (((2 * qd + 1) ^ r8) << 4), u[nt][4], u[nt][5], u[nt][6], u[nt][7]);
    }
    // the two n-tiles' accumulation chains are interleaved to hide MMA latency
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const uint32_t b0 = e4m3x2_to_f16x2(static_cast<uint16_t>(u[nt][ks] & 0xffffu));
        const uint32_t b1 = e4m3x2_to_f16x2(static_cast<uint16_t>(u[nt][ks] >> 16));
        mma_f16(s[nt], qa[ks], b0, b1);
      }
    }
  }
}

// O[16 rows x 128] += P[16 x 16 keys] V for the warp's keys of the page in `vt`.
template <int KV>
__device__ __forceinline__ void pv(float (&o)[16][4], const uint32_t (&pa)[4], uint32_t vt,
                                   int w, int lane) {
  if (KV == HPA_KV_BF16) {
    const int mi = lane >> 3, key = 16 * w + (mi & 1) * 8 + (lane & 7);
    const uint32_t row = vt + key * 128;
#pragma unroll
    for (int np = 0; np < 8; ++np) {
      const int chunk = (np & 3) * 2 + (mi >> 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(row + (np >> 2) * 8192 + ((chunk ^ (lane & 7)) << 4), b0, b1, b2, b3);
      mma_bf16(o[2 * np], pa, b0, b1);
      mma_bf16(o[2 * np + 1], pa, b2, b3);
    }
  } else {
    // thread (r8 = c, qd) reads dims [16c, 16c+16) of keys 2qd, 2qd+1, 2qd+8, 2qd+9;
    // output column n of n-tile i is head dim 16 n + i.
    const int c = lane >> 2, qd = lane & 3;
    uint32_t R[4][4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int key = 16 * w + 2 * qd + (k & 1) + (k >> 1) * 8;
      lds128(vt + key * 128 + ((c ^ (key & 7)) << 4), R[k][0], R[k][1], R[k][2], R[k][3]);
    }
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {  // byte pairs (0,1) and (2,3) of the word
        // bytes [k0.b, k1.b, k0.b+1, k1.b+1] for b = 2*hb
        const uint32_t sel = hb ? 0x7362u : 0x5140u;
        const uint32_t lo01 = __byte_perm(R[0][wd], R[1][wd], sel);
        const uint32_t lo23 = __byte_perm(R[2][wd], R[3][wd], sel);
        const int i = 4 * wd + 2 * hb;
        mma_f16(o[i], pa, e4m3x2_to_f16x2(static_cast<uint16_t>(lo01 & 0xffffu)),
                e4m3x2_to_f16x2(static_cast<uint16_t>(lo23 & 0xffffu)));
        mma_f16(o[i + 1], pa, e4m3x2_to_f16x2(static_cast<uint16_t>(lo01 >> 16)),
                e4m3x2_to_f16x2(static_cast<uint16_t>(lo23 >> 16)));
      }
    }
  }
}

__device__ __forceinline__ void store_bf16x4(__nv_bfloat16 *dst, float4 v) {
  uint2 pk;
  pk.x = pack_bf16(v.x, v.y);
  pk.y = pack_bf16(v.z, v.w);
  *reinterpret_cast<uint2 *>(dst) = pk;
}

// Fused combine by the last-arriving CTA: log-sum-exp merge of segments
// [seg_first, seg_first + nseg) of request r for the G * q_len rows of KV head h,
// read through L2 (other CTAs wrote them), written as the final bf16 output.
template <int KV>
__device__ void merge_request(const AttnParams &p, int r, int h, int seg_first, int nseg,
                              int tid) {
  const int G = p.G, q_len = p.q_len, rb = row_base();
  const int64_t per_seg = static_cast<int64_t>(q_len) * p.Hq;
  for (int v = tid; v < group_rows(p) * (HEAD_DIM / 4); v += kConsumerWarps * 32) {
    const int row = rb + v / (HEAD_DIM / 4), c4 = v % (HEAD_DIM / 4);
    const int64_t col = static_cast<int64_t>(row / G) * p.Hq + h * G + row % G;
    float M = -CUDART_INF_F;
    for (int i = 0; i < nseg; ++i) M = fmaxf(M, __ldcg(p.partial_lse + (seg_first + i) * per_seg + col));
    const float Mb = M == -CUDART_INF_F ? 0.f : M;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float W = 0.f;
    for (int i0 = 0; i0 < nseg; i0 += 4) {
      float l[4];
      float4 o[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i0 + u < nseg) {
          const int64_t sr = (seg_first + i0 + u) * per_seg + col;
          l[u] = __ldcg(p.partial_lse + sr);
          o[u] = __ldcg(reinterpret_cast<const float4 *>(p.partial_o + sr * HEAD_DIM) + c4);
        }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i0 + u < nseg) {
          const float wt = expf(l[u] - Mb);
          acc.x += wt * o[u].x;
          acc.y += wt * o[u].y;
          acc.z += wt * o[u].z;
          acc.w += wt * o[u].w;
          W += wt;
        }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    const int64_t orow = (static_cast<int64_t>(r) * per_seg + col) * HEAD_DIM;
    store_bf16x4(p.out + orow + 4 * c4,
                 make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
    if (c4 == 0 && p.out_lse != nullptr)
      p.out_lse[static_cast<int64_t>(r) * per_seg + col] = W > 0.f ? Mb + logf(W) : -CUDART_INF_F;
  }
}

// ----------------------------------------------------------------------------- consumer
template <int KV, bool FUSED, bool ALLH>
__device__ void consumer(const AttnParams &p, uint8_t *smem, int s_begin, int s_end, int tile,
                         int h0) {
  using S = Smem<KV>;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r8 = lane >> 2, qd = lane & 3;
  const uint32_t base = smem_u32(smem);
  const uint32_t full0 = base + S::kBars, empty0 = full0 + 8 * S::kStages;
  float *mbuf = reinterpret_cast<float *>(smem + S::kMerge);
  float *sm_m = reinterpret_cast<float *>(smem + S::kStats);
  float *sm_l = sm_m + kConsumerWarps * MAX_ROWS;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kFlag);

  // rows of this CTA's group: local index row, global query row rb + row
  const int G = p.G, rows = group_rows(p), q_len = p.q_len, rb = row_base();
  const int row0 = r8, row1 = r8 + 8;
  const bool v0 = row0 < rows, v1 = row1 < rows;
  const int j0 = (rb + row0) / G, j1 = (rb + row1) / G;

  const uint32_t qfull0 = empty0 + 8 * S::kStages, qempty0 = qfull0 + 16;
  int stage = 0;
  uint32_t phase = 0;
  // score and output scales of the KV head (loaded once on the per-head grid)
  float sl2_h = p.scale_log2, vsc_h = 1.f;
  if (!ALLH && KV == HPA_KV_E4M3) {
    sl2_h *= p.k_scale[h0];
    vsc_h = p.v_scale[h0];
  }
  const int hpc = ALLH ? p.heads_per_cta : 1, n_items = (s_end - s_begin) * hpc;
  for (int k = 0; k < n_items; ++k) {
    const int s = s_begin + k / hpc, h = h0 + k % hpc, slot = k & 1;
    float sl2 = sl2_h, vsc = vsc_h;
    if (ALLH && KV == HPA_KV_E4M3) {
      sl2 *= p.k_scale[h];
      vsc = p.v_scale[h];
    }
    bool ok = !*abort_flag && mbar_wait_bounded(qfull0 + 8 * slot, (k >> 1) & 1);
    ok = __all_sync(kFull, ok);
    SegInfo f;
    {
      const int4 inf = reinterpret_cast<const int4 *>(smem + S::kInfo)[2 * slot];
      f.r = inf.x;
      f.L = inf.y;
      f.klo = inf.z;
      f.khi = inf.w;
      f.pg0 = f.klo / PAGE;
      f.pg1 = ok ? (f.khi + PAGE - 1) / PAGE : f.pg0;  // no pages if the wait gave up
    }
    if (ok && f.L < q_len && w == 0 && lane == 0) status_or(p.tm, HPA_STATUS_BAD_SEQLEN);
    // fused combine: first segment and segment count of this request
    int seg_first = 0, nseg = 0;
    if (FUSED) {
      const int4 inf2 = reinterpret_cast<const int4 *>(smem + S::kInfo)[2 * slot + 1];
      seg_first = inf2.x;
      nseg = inf2.y;
    }
    const int lim_min = f.L - q_len + 1;  // first key hidden from some row
    const int lim0 = v0 ? f.L - q_len + 1 + j0 : f.L;
    const int lim1 = v1 ? f.L - q_len + 1 + j1 : f.L;

    // query fragments (A operand, 16 rows x 128) from the staged rows
    uint32_t qa[8][4];
    // per-row score factors: sm_scale * log2 e (* k scale), times 2^-e_row on the E4M3 path
    float sl2_0 = sl2, sl2_1 = sl2;
    {
      const uint8_t *qs = smem + S::kQ + slot * kQSlotBytes;
      const __nv_bfloat16 *q0 = reinterpret_cast<const __nv_bfloat16 *>(qs + row0 * kQRowBytes);
      const __nv_bfloat16 *q1 = reinterpret_cast<const __nv_bfloat16 *>(qs + row1 * kQRowBytes);
      // E4M3 path: the query enters f16 MMAs.  Each row is scaled by 2^e_row so that its
      // largest |element| lands in [2^14, 2^15): a bf16 value that large or small (up to
      // ~3e38 or down to bf16's subnormals) cannot overflow f16 or lose bits to f16
      // subnormals, since every element within 2^-28 of the row maximum stays an f16
      // normal and converts exactly.  The factor is taken back out of the scores.
      float qsc0 = 1.f, qsc1 = 1.f;
      if (KV == HPA_KV_E4M3) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {  // this thread's 32 dims of each row
          const int d0 = 32 * qd + 4 * ks;
          if (v0) a0 = fmaxf(a0, absmax4_bf16(q0 + d0));
          if (v1) a1 = fmaxf(a1, absmax4_bf16(q1 + d0));
        }
        a0 = fmaxf(a0, __shfl_xor_sync(kFull, a0, 1));  // the 4 threads of a row (qd)
        a0 = fmaxf(a0, __shfl_xor_sync(kFull, a0, 2));
        a1 = fmaxf(a1, __shfl_xor_sync(kFull, a1, 1));
        a1 = fmaxf(a1, __shfl_xor_sync(kFull, a1, 2));
        const int e0 = f16_row_exponent(a0), e1 = f16_row_exponent(a1);
        qsc0 = exp2i(e0);
        qsc1 = exp2i(e1);
        sl2_0 = sl2 * exp2i(-e0);
        sl2_1 = sl2 * exp2i(-e1);
      }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        if (KV == HPA_KV_BF16) {
          const int d0 = 16 * ks + 2 * qd;
          qa[ks][0] = v0 ? *reinterpret_cast<const uint32_t *>(q0 + d0) : 0u;
          qa[ks][1] = v1 ? *reinterpret_cast<const uint32_t *>(q1 + d0) : 0u;
          qa[ks][2] = v0 ? *reinterpret_cast<const uint32_t *>(q0 + d0 + 8) : 0u;
          qa[ks][3] = v1 ? *reinterpret_cast<const uint32_t *>(q1 + d0 + 8) : 0u;
        } else {
          const int d0 = 32 * qd + 4 * ks;
          auto h2 = [](const __nv_bfloat16 *x, float sc) {
            const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(x));
            return pack_f16(t.x * sc, t.y * sc);
          };
          qa[ks][0] = v0 ? h2(q0 + d0, qsc0) : 0u;
          qa[ks][1] = v1 ? h2(q1 + d0, qsc1) : 0u;
          qa[ks][2] = v0 ? h2(q0 + d0 + 2, qsc0) : 0u;
          qa[ks][3] = v1 ? h2(q1 + d0 + 2, qsc1) : 0u;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(qempty0 + 8 * slot);  // the slot may be refilled

    float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[i][e] = 0.f;

    for (int pg = f.pg0; pg < f.pg1; ++pg) {
      const bool got = !(*abort_flag) && mbar_wait_bounded(full0 + 8 * stage, phase);
      if (!__all_sync(kFull, got)) {
        ok = false;  // the rest of this CTA's work is abandoned (see below)
        break;
      }
      uint8_t *kt = smem + stage * S::kStageBytes;
      uint8_t *vt = kt + Cfg<KV>::kKBytes;
      const int key0 = pg * PAGE, wk = key0 + 16 * w;
      const bool tail = wk + 16 > f.L;
      if (tail) {
        zero_tail_rows<KV>(vt, w, wk, f.L, lane);
        __syncwarp();
      }

      float sc[2][4];
      qk<KV>(sc, qa, smem_u32(kt), w, lane);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[nt][e] *= e < 2 ? sl2_0 : sl2_1;
      if (wk + 16 > lim_min) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int key = wk + 8 * nt + 2 * qd + (e & 1);
            if (key >= (e < 2 ? lim0 : lim1)) sc[nt][e] = -CUDART_INF_F;
          }
      }
      // online softmax, rows row0 (e = 0,1) and row1 (e = 2,3)
      float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
      float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 2));
      // Conditional rescale: the reference max m moves only when a score exceeds it
      // by more than kRescaleSlack (base 2), so p = 2^(s - m) <= 2^kRescaleSlack and
      // O / l keep one consistent reference; exact up to rounding, and the O rescale
      // below is almost always skipped after a segment's first pages.
      const float mn0 = mx0 > m0 + kRescaleSlack ? mx0 : m0;
      const float mn1 = mx1 > m1 + kRescaleSlack ? mx1 : m1;
      const float b0 = mn0 == -CUDART_INF_F ? 0.f : mn0;
      const float b1 = mn1 == -CUDART_INF_F ? 0.f : mn1;
      const float a0 = exp2f(m0 - b0), a1 = exp2f(m1 - b1);
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        sc[nt][0] = exp2f(sc[nt][0] - b0);
        sc[nt][1] = exp2f(sc[nt][1] - b0);
        sc[nt][2] = exp2f(sc[nt][2] - b1);
        sc[nt][3] = exp2f(sc[nt][3] - b1);
      }
      l0 = l0 * a0 + (sc[0][0] + sc[0][1] + sc[1][0] + sc[1][1]);
      l1 = l1 * a1 + (sc[0][2] + sc[0][3] + sc[1][2] + sc[1][3]);
      // skip the rescale when no row of this warp moved its reference (alpha == 1)
      if (__any_sync(kFull, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          o[i][0] *= a0;
          o[i][1] *= a0;
          o[i][2] *= a1;
          o[i][3] *= a1;
        }
      }
      uint32_t pa[4];
      if (KV == HPA_KV_BF16) {
        pa[0] = pack_bf16(sc[0][0], sc[0][1]);
        pa[1] = pack_bf16(sc[0][2], sc[0][3]);
        pa[2] = pack_bf16(sc[1][0], sc[1][1]);
        pa[3] = pack_bf16(sc[1][2], sc[1][3]);
      } else {
        pa[0] = pack_f16(sc[0][0], sc[0][1]);
        pa[1] = pack_f16(sc[0][2], sc[0][3]);
        pa[2] = pack_f16(sc[1][0], sc[1][1]);
        pa[3] = pack_f16(sc[1][2], sc[1][3]);
      }
      pv<KV>(o, pa, smem_u32(vt), w, lane);
      __syncwarp();
      if (tail) fence_proxy_async_smem();  // generic writes before the next TMA fill
      if (lane == 0) mbar_arrive(empty0 + 8 * stage);
      if (++stage == S::kStages) {
        stage = 0;
        phase ^= 1;
      }
    }
    // A timed-out warp flags the map and raises the CTA's abort flag; it still
    // takes part in the epilogue's named barriers below so that no other
    // consumer warp waits on it.  Later waits see the flag and fail at once.
    if (!ok && lane == 0) {
      status_or(p.tm, HPA_STATUS_TIMEOUT);
      *abort_flag = 1;
    }

    // ---- segment end: merge the four warps' (m, l, O) and store the partial
    l0 += __shfl_xor_sync(kFull, l0, 1);
    l0 += __shfl_xor_sync(kFull, l0, 2);
    l1 += __shfl_xor_sync(kFull, l1, 1);
    l1 += __shfl_xor_sync(kFull, l1, 2);
    if (qd == 0) {
      sm_m[w * MAX_ROWS + row0] = m0;
      sm_l[w * MAX_ROWS + row0] = l0;
      sm_m[w * MAX_ROWS + row1] = m1;
      sm_l[w * MAX_ROWS + row1] = l1;
    }
    named_barrier(1, kConsumerWarps * 32);
    auto row_stats = [&](int row, float &M, float &Lsum) {
      M = -CUDART_INF_F;
#pragma unroll
      for (int x = 0; x < kConsumerWarps; ++x) M = fmaxf(M, sm_m[x * MAX_ROWS + row]);
      const float Mb = M == -CUDART_INF_F ? 0.f : M;
      Lsum = 0.f;
#pragma unroll
      for (int x = 0; x < kConsumerWarps; ++x)
        Lsum += sm_l[x * MAX_ROWS + row] * exp2f(sm_m[x * MAX_ROWS + row] - Mb);
      M = Mb;
    };
    float M0, L0, M1, L1;
    row_stats(row0, M0, L0);
    row_stats(row1, M1, L1);
    const float f0 = L0 > 0.f ? exp2f(m0 - M0) / L0 * vsc : 0.f;
    const float f1 = L1 > 0.f ? exp2f(m1 - M1) / L1 * vsc : 0.f;
    constexpr int MS = S::kMergeStride;
    float *mine = mbuf + (w & 1) * (MAX_ROWS * MS);
    // one merge pass: warps 0 / 1 store (ADD = false), then warps 2 / 3 add
    auto merge = [&](auto add_tag) {
      constexpr bool ADD = decltype(add_tag)::value;
      if (KV == HPA_KV_BF16) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int pos = i * 8 + 2 * qd;
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            if (hr == 0 ? !v0 : !v1) continue;
            float2 *d = reinterpret_cast<float2 *>(mine + (hr ? row1 : row0) * MS + pos);
            const float fs = hr ? f1 : f0;
            float2 nv = make_float2(o[i][2 * hr] * fs, o[i][2 * hr + 1] * fs);
            if (ADD) {
              const float2 t = *d;
              nv.x += t.x;
              nv.y += t.y;
            }
            *d = nv;
          }
        }
      } else {
        // o[i][c] of row hr holds dim 32 qd + 16 (c & 1) + i
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          if (hr == 0 ? !v0 : !v1) continue;
          const float fs = hr ? f1 : f0;
          float *rowp = mine + (hr ? row1 : row0) * MS;
#pragma unroll
          for (int half = 0; half < 2; ++half)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              float4 *d = reinterpret_cast<float4 *>(rowp + merge_phys(32 * qd + 16 * half + 4 * k));
              const int c = 2 * hr + half;
              float4 nv = make_float4(o[4 * k][c] * fs, o[4 * k + 1][c] * fs,
                                      o[4 * k + 2][c] * fs, o[4 * k + 3][c] * fs);
              if (ADD) {
                const float4 t = *d;
                nv.x += t.x;
                nv.y += t.y;
                nv.z += t.z;
                nv.w += t.w;
              }
              *d = nv;
            }
        }
      }
    };
    if (w < 2) merge(std::false_type());
    named_barrier(1, kConsumerWarps * 32);
    if (w >= 2) merge(std::true_type());
    named_barrier(1, kConsumerWarps * 32);
    const int tid = threadIdx.x;
    // fused combine, single-segment request: this segment is the whole result
    const bool direct = FUSED && nseg == 1;
    for (int v = tid; v < rows * (HEAD_DIM / 4); v += kConsumerWarps * 32) {
      const int row = v / (HEAD_DIM / 4), c4 = v % (HEAD_DIM / 4);
      const int j = (rb + row) / G, g = (rb + row) % G;
      const int64_t dst = ((static_cast<int64_t>(direct ? f.r : s) * q_len + j) * p.Hq + h * G + g) *
                          HEAD_DIM;
      const float *ra = mbuf + row * MS;           // buffer A
      const float *rb2 = ra + MAX_ROWS * MS;         // buffer B
      const int pos = KV == HPA_KV_BF16 ? 4 * c4 : merge_phys(4 * c4);
      const float4 a = *reinterpret_cast<const float4 *>(ra + pos);
      const float4 b = *reinterpret_cast<const float4 *>(rb2 + pos);
      const float4 val = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
      if (direct)
        store_bf16x4(p.out + dst + 4 * c4, val);
      else
        reinterpret_cast<float4 *>(p.partial_o + dst)[c4] = val;
    }
    if (tid < rows) {
      float M, Lsum;
      row_stats(tid, M, Lsum);
      const int j = (rb + tid) / G, g = (rb + tid) % G;
      const float lse = Lsum > 0.f ? (M + log2f(Lsum)) * 0.69314718055994531f : -CUDART_INF_F;
      if (!direct)
        p.partial_lse[(static_cast<int64_t>(s) * q_len + j) * p.Hq + h * G + g] = lse;
      else if (p.out_lse != nullptr)
        p.out_lse[(static_cast<int64_t>(f.r) * q_len + j) * p.Hq + h * G + g] = lse;
    }
    if (FUSED && !direct) {  // CTA-uniform: all consumer warps take the barriers
      // Fused combine: count this partial in; the CTA that brings the count to
      // nseg merges all of the request's partials for this KV head.  Nobody waits:
      // every other CTA just moves on.
      __threadfence();  // this CTA's partial stores before its arrival
      named_barrier(1, kConsumerWarps * 32);
      volatile int *last = reinterpret_cast<volatile int *>(smem + S::kFlag + 4);
      int32_t *counter = p.arrivals + (static_cast<int64_t>(f.r) * p.Hkv + h) * gridDim.z + blockIdx.z;
      if (tid == 0) *last = atomicAdd(counter, 1) == nseg - 1;
      named_barrier(1, kConsumerWarps * 32);
      if (*last) {
        __threadfence();
        merge_request<KV>(p, f.r, h, seg_first, nseg, tid);
        if (tid == 0) *counter = 0;  // ready for the next call
      }
    }
    named_barrier(1, kConsumerWarps * 32);
  }
}

// ----------------------------------------------------------------------------- kernel
template <int KV, bool FUSED, bool ALLH>
__global__ void __launch_bounds__(kThreads, 2)
    decode_attn_kernel(const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const AttnParams p) {
  using S = Smem<KV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int c = blockIdx.x, h0 = ALLH ? 0 : blockIdx.y;  // first KV head of the CTA
  __shared__ int hdr[5];  // go, tile, s_begin, s_end, bad map -- read once, used by all threads
  const uint32_t base = smem_u32(smem);
  unsigned long long *trace =
      p.trace ? p.trace + 4 * ((static_cast<int64_t>(blockIdx.z) * gridDim.y + blockIdx.y) * p.C + c)
              : nullptr;
  if (trace && threadIdx.x == 0) trace[0] = globaltimer_ns();
  // Nothing above this line reads memory that an earlier kernel writes: with
  // programmatic dependent launch the prologue overlaps the previous kernel.
  pdl_wait();
  if (threadIdx.x == 0) {
    const int32_t *tm = p.tm;
    const int tile = tm[TM_TILE];
    int go = tm[TM_STATUS] == 0;
    if (go && (tm[TM_B] != p.B || tm[TM_C] != p.C || tile <= 0 || tile % PAGE != 0)) {
      if (c == 0 && h0 == 0) status_or(p.tm, HPA_STATUS_MISMATCH);
      go = 0;
    }
    if (go && !map_ranges_ok(tm, p.lay, p.B, p.C, c)) {
      status_or(p.tm, HPA_STATUS_BAD_MAP);
      go = 0;
    }
    hdr[4] = !go;
    hdr[1] = tile;
    hdr[2] = go ? tm[p.lay.cta_seg + c] : 0;
    hdr[3] = go ? tm[p.lay.cta_seg + c + 1] : 0;
    hdr[0] = go && hdr[2] < hdr[3];
    for (int st = 0; st < S::kStages; ++st) {
      mbar_init(base + S::kBars + 8 * st, 1);
      mbar_init(base + S::kBars + 8 * (S::kStages + st), kConsumerWarps);
    }
    for (int sl = 0; sl < 2; ++sl) {
      mbar_init(base + S::kBars + 8 * (2 * S::kStages + sl), 32);                 // qfull
      mbar_init(base + S::kBars + 8 * (2 * S::kStages + 2 + sl), kConsumerWarps);  // qempty
    }
    *reinterpret_cast<int *>(smem + S::kFlag) = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();  // the combine kernel may be scheduled; it waits for this grid
  if (trace && threadIdx.x == 0) {
    trace[1] = globaltimer_ns();
    trace[3] = smid() | (static_cast<unsigned long long>(hdr[3] - hdr[2]) << 32);
  }
  if (!hdr[0]) {  // bad map, or a partition with no tiles
    if (FUSED && hdr[4]) {
      // fused combine on a bad map: NaN outputs, as the combine kernel writes;
      // CTA (c, h) covers requests c, c + C, ... for the query heads of its KV heads
      const float nan = CUDART_NAN_F;
      for (int r = c; r < p.B; r += p.C)
        for (int v = threadIdx.x; v < (ALLH ? p.Hkv : 1) * group_rows(p) * (HEAD_DIM / 4);
             v += kThreads) {
          const int hh = h0 + v / (group_rows(p) * (HEAD_DIM / 4));
          const int vr = v % (group_rows(p) * (HEAD_DIM / 4));
          const int row = row_base() + vr / (HEAD_DIM / 4), c4 = vr % (HEAD_DIM / 4);
          const int64_t col = static_cast<int64_t>(row / p.G) * p.Hq + hh * p.G + row % p.G;
          const int64_t orow = static_cast<int64_t>(r) * p.q_len * p.Hq + col;
          store_bf16x4(p.out + orow * HEAD_DIM + 4 * c4, make_float4(nan, nan, nan, nan));
          if (c4 == 0 && p.out_lse != nullptr) p.out_lse[orow] = nan;
        }
    }
    if (trace && threadIdx.x == 0) trace[2] = globaltimer_ns();
    return;
  }
  const int tile = hdr[1], s_begin = hdr[2], s_end = hdr[3];

  if (threadIdx.x >= kConsumerWarps * 32) {
    producer<KV, FUSED, ALLH>(p, &tmk, &tmv, smem, s_begin, s_end, tile, h0);
  } else {
    consumer<KV, FUSED, ALLH>(p, smem, s_begin, s_end, tile, h0);
    if (trace && threadIdx.x == 0) trace[2] = globaltimer_ns();  // after the last epilogue
  }
}

template <int KV, bool FUSED, bool ALLH>
cudaError_t launch(const AttnParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                   cudaStream_t s) {
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(decode_attn_kernel<KV, FUSED, ALLH>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<KV>::kAlloc);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.C, ALLH ? 1 : p.Hkv, (p.rows + MAX_ROWS - 1) / MAX_ROWS);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Smem<KV>::kAlloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_attn_kernel<KV, FUSED, ALLH>, tmk, tmv, p);
}

template <int KV>
int occupancy(int *ctas) {
  cudaError_t e = cudaFuncSetAttribute(decode_attn_kernel<KV, false, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Smem<KV>::kAlloc);
  if (e != cudaSuccess) return -1;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, decode_attn_kernel<KV, false, false>,
                                                    kThreads, Smem<KV>::kAlloc);
  return e == cudaSuccess ? 0 : -1;
}

}  // namespace

cudaError_t launch_decode_attn(const AttnParams &p, const CUtensorMap &tmk,
                               const CUtensorMap &tmv, int kv_dtype, cudaStream_t s) {
  const bool fused = p.out != nullptr;  // the fused combine is its own instantiation
  const bool all_heads = p.heads_per_cta > 1;  // every KV head in the CTA (unfused only)
  if (fused && all_heads) return cudaErrorInvalidValue;
  if (kv_dtype == HPA_KV_BF16)
    return fused       ? launch<HPA_KV_BF16, true, false>(p, tmk, tmv, s)
           : all_heads ? launch<HPA_KV_BF16, false, true>(p, tmk, tmv, s)
                       : launch<HPA_KV_BF16, false, false>(p, tmk, tmv, s);
  return fused       ? launch<HPA_KV_E4M3, true, false>(p, tmk, tmv, s)
         : all_heads ? launch<HPA_KV_E4M3, false, true>(p, tmk, tmv, s)
                     : launch<HPA_KV_E4M3, false, false>(p, tmk, tmv, s);
}

int attn_ctas_per_sm(int kv_dtype, int q_len, int *ctas) {
  (void)q_len;
  return kv_dtype == HPA_KV_BF16 ? occupancy<HPA_KV_BF16>(ctas) : occupancy<HPA_KV_E4M3>(ctas);
}

}  // namespace hpa
