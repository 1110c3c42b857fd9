// Internal declarations shared by the CUDA translation units of libhpa:
// task map layout, launch parameter blocks, and thin inline-PTX wrappers
// (mbarrier, TMA tensor copies, ldmatrix, mma.sync) for sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "hpa.h"

namespace hpa {

// ----------------------------------------------------------------------------- task map
enum : int {
  TM_T = 0, TM_BASE, TM_REM, TM_C, TM_B, TM_S, TM_STATUS, TM_TILE, TM_KIND, TM_SPLITS,
  TM_SCAP, TM_HEADER_WORDS = 16
};

struct TaskMapLayout {
  int64_t lens, cu_tiles, cta_begin, cta_seg, seg_off, segs;  // word offsets
  __host__ __device__ static TaskMapLayout make(int64_t B, int64_t C) {
    TaskMapLayout t;
    t.lens = TM_HEADER_WORDS;
    t.cu_tiles = t.lens + B;
    t.cta_begin = t.cu_tiles + B + 1;
    t.cta_seg = t.cta_begin + C + 1;
    t.seg_off = t.cta_seg + C + 1;
    t.segs = (t.seg_off + B + 1 + 3) & ~int64_t(3);  // 16-byte aligned rows
    return t;
  }
  __host__ __device__ int64_t words(int64_t s_cap) const { return segs + 4 * s_cap; }
};

constexpr int PAGE = 64;       // tokens per KV page
constexpr int HEAD_DIM = 128;  // d
constexpr int MAX_ROWS = 16;   // query rows per CTA (one m16 MMA tile)
constexpr int MAX_ROWS_TOTAL = 64;  // G * q_len rows per KV head, in groups of 16

// ----------------------------------------------------------------------------- launch blocks
struct AttnParams {
  const __nv_bfloat16 *q;
  int32_t *tm;
  const int32_t *page_indptr, *page_indices;
  const float *k_scale, *v_scale;
  float *partial_o, *partial_lse;
  unsigned long long *trace;  // optional: 4 words per CTA (entry, go, end, smid | segs << 32)
  __nv_bfloat16 *out;         // fused combine: final output (nullptr: write partials only)
  float *out_lse;             // fused combine: final lse (optional)
  int32_t *arrivals;          // fused combine: [B][Hkv] arrival counters, zero between calls
  int64_t num_pages;
  TaskMapLayout lay;
  int B, C, q_len, Hq, Hkv, G, rows;
  int heads_per_cta;  // KV heads one CTA walks per segment: 1 (grid over heads) or Hkv
  float scale_log2;   // sm_scale * log2(e)
};

// Records e as the calling thread's last CUDA error (hpa_last_cuda_error) and
// returns HPA_ERR_CUDA; every entry point reports runtime failures through it.
int cuda_fail(cudaError_t e);
int last_cuda_error();

constexpr size_t kPlanStageLimit = 40 * 1024;  // shared memory the plan kernel may stage in
size_t plan_stage_bytes(int B, int C, int kind);
cudaError_t launch_plan(const int32_t *seq_lens, int B, int tile, int C, int kind, int splits,
                        int32_t *tm, int64_t s_cap, cudaStream_t s);
cudaError_t launch_combine(const float *po, const float *plse, int32_t *tm, int B, int C,
                           int q_len, int Hq, __nv_bfloat16 *out, float *out_lse,
                           cudaStream_t s);
cudaError_t launch_decode_attn(const AttnParams &p, const CUtensorMap &tmk,
                               const CUtensorMap &tmv, int kv_dtype, cudaStream_t s);
int attn_ctas_per_sm(int kv_dtype, int q_len, int *ctas);  // occupancy query (host)
cudaError_t launch_decode_attn_tc(const AttnParams &p, const CUtensorMap &tmk,
                                  const CUtensorMap &tmv, int kv_dtype, cudaStream_t s);
int attn_tc_ctas_per_sm(int kv_dtype, int rows, int *ctas);  // occupancy query (host)
cudaError_t launch_selftest_wait(int32_t *status, long long limit_ns, cudaStream_t s);

struct StoreKvParams {
  const __nv_bfloat16 *k_new, *v_new;
  const int32_t *seq_lens, *page_indptr, *page_indices;
  int64_t num_pages;
  const float *cos_sin;
  int max_pos;
  const float *norm_w;
  float eps;
  int use_hadamard, kv_dtype;
  const float *k_scale, *v_scale;
  void *k_pool, *v_pool;
  int B, q_len, Hkv;
  int32_t *status;
};
cudaError_t launch_store_kv(const StoreKvParams &p, cudaStream_t s);

// ----------------------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint32_t smid() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on an mbarrier phase: gives up after ~limit_ns and returns false.
// kRolled keeps the 64-retry loop between clock checks rolled: a few instructions at
// each call site instead of 64 unrolled retries, for kernels whose hot loops hold many
// waits (the tcgen05 attention kernel: 1974 -> 1872 us at 64 rows; the mma.sync
// kernel was 2 % slower with it, so it keeps the unrolled form).
template <bool kRolled>
__device__ __forceinline__ bool mbar_wait_bounded_impl(uint32_t bar, uint32_t parity,
                                                       uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if constexpr (kRolled) {
#pragma unroll 1
      for (int i = 0; i < 64; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    } else {
      for (int i = 0; i < 64; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    }
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns = 2000000000ull) {
  return mbar_wait_bounded_impl<false>(bar, parity, limit_ns);
}
__device__ __forceinline__ bool mbar_wait_bounded_rolled(uint32_t bar, uint32_t parity,
                                                         uint64_t limit_ns = 2000000000ull) {
  return mbar_wait_bounded_impl<true>(bar, parity, limit_ns);
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 3-D tiled TMA load global -> shared, completion counted on `bar` (bytes).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                            int x, int y, int z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                        uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                          uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void lds128(uint32_t addr, uint32_t &a, uint32_t &b, uint32_t &c,
                                       uint32_t &d) {
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
               : "r"(addr));
}

// D += A(16x16, row) * B(16x8, col); bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Same with fp16 inputs.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (lo, hi) fp32 -> two E4M3 codes, lo in the low byte; round to nearest even,
// saturating at +-448.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 codes (low 16 bits of `v`, element 0 in the low byte) -> f16x2 with
// element 0 in the low half (exact: every E4M3 value is an f16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Two fp32 values in one 64-bit register for the packed FP32 pipe of sm_100-family
// SMs (fma/add/sub/mul .f32x2): each half is rounded exactly as the scalar operation
// would round it, and one instruction does both.  pk(a, b) puts a in the low half.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pk(float a, float b) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk(f32x2 v, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// 2^k for an integer k in [-126, 127], built from the exponent bits (exact).
__device__ __forceinline__ float exp2i(int k) {
  return __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Programmatic dependent launch: a grid launched with programmatic stream
// serialisation may start before its predecessor ends; pdl_wait() blocks until
// the predecessor grids have completed and their writes are visible (a no-op
// when the grid was launched without the attribute).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void status_or(int32_t *tm, int bits) {
  atomicOr(reinterpret_cast<int *>(tm + TM_STATUS), bits);
}

// One segment row of a task map, checked before use: request in [0, B), owned by
// partition c, 0 <= tile_lo < tile_hi <= ceil(L_r / tile).  A row that fails (a
// map corrupted after hpa_plan wrote it) is reported as HPA_STATUS_BAD_MAP when
// `report` is set and read as an empty segment of request 0, so no kernel follows
// an index out of the buffers the map was sized for.  Every reader of a row gets
// the same answer, so the roles of one CTA stay in step.
struct SegRow {
  int r, L, klo, khi;  // request, its length, key range [klo, khi)
};
__device__ __forceinline__ SegRow read_seg_row(int32_t *tm, const TaskMapLayout &lay, int B,
                                               int s, int c, int tile, bool report) {
  const int4 sg = reinterpret_cast<const int4 *>(tm + lay.segs)[s];
  if (sg.x >= 0 && sg.x < B && sg.w == c && sg.y >= 0 && sg.y < sg.z) {
    const int L = tm[lay.lens + sg.x];
    if (L >= 1 && sg.z <= (L - 1) / tile + 1) {
      const long long hi = static_cast<long long>(sg.z) * tile;
      return SegRow{sg.x, L, sg.y * tile, hi < L ? static_cast<int>(hi) : L};
    }
  }
  if (report) status_or(tm, HPA_STATUS_BAD_MAP);
  return SegRow{0, 1 << 30, 0, 0};
}

// Header checks an attention kernel makes before it walks partition c: the map's
// kind and segment capacity match what hpa_plan / hpa_plan_static build for (B, C),
// and c's segment range lies inside the map's S segments.
__device__ __forceinline__ bool map_ranges_ok(const int32_t *tm, const TaskMapLayout &lay, int B,
                                              int C, int c) {
  const int kind = tm[TM_KIND], S = tm[TM_S];
  const int cap = kind == 1 ? C : B + C - 1;
  const int sb = tm[lay.cta_seg + c], se = tm[lay.cta_seg + c + 1];
  return kind >= 0 && kind <= 2 && tm[TM_SCAP] == cap && S >= 0 && S <= cap && sb >= 0 &&
         sb <= se && se <= S;
}

}  // namespace hpa
