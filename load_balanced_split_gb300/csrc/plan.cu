// Task Assign: builds the split-KV task map on the device with one CTA.
//
// Dynamic map ("Hy3 Preview AI Infra 推理优化精读笔记", §3.1 方案 steps 1-4;
// "大模型推理性能优化新范式：Hy3架构下的全栈优化技术拆解", §二.1 budget rule):
//   n_r = ceil(L_r / tile), cu_tiles = exclusive scan of n_r, T = cu_tiles[B],
//   base = T / C, rem = T % C, partition c owns stream tiles
//   [c*base + min(c, rem), (c+1)*base + min(c+1, rem)) -- a greedy fill of
//   equal budgets along the request-major tile stream -- and its range is
//   cut at request boundaries into segments.
// Static map (the fixed split-KV the same §3.1 contrasts it with): request r
//   is cut into min(splits, n_r) near-equal chunks, partition r*splits+s owns
//   chunk s.
// Token-weighted map (kind 2): the same contiguous partitions of the tile
//   stream, with budgets in keys: tile t (keys P_t before it, w_t in it) goes
//   to partition floor(C (2 P_t + w_t) / (2 K)), K the total key count, so a
//   partial last tile weighs its fill.
#include <climits>

#include "hpa_internal.cuh"

namespace hpa {
namespace {

// The plan is latency-bound: one CTA, a few dependent rounds.  Its block size is
// the smallest of 32 / 128 / 256 / 1024 threads that gives every request and
// every partition a thread of its own (1024 beyond that, looping), so small
// batches pay for few warps in each block-wide scan and barrier.

// Inclusive scan over the block; `total` receives the block-wide sum.
template <int kPlanThreads>
__device__ long long block_scan(long long v, long long *wbuf, long long &total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int o = 1; o < 32; o <<= 1) {
    long long n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  constexpr int kWarps = kPlanThreads / 32;  // wbuf holds one partial sum per warp
  if (lane == 31) wbuf[wid] = v;
  __syncthreads();
  if (wid == 0) {
    long long w = lane < kWarps ? wbuf[lane] : 0;
    for (int o = 1; o < kWarps; o <<= 1) {
      long long n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    if (lane < kWarps) wbuf[lane] = w;
  }
  __syncthreads();
  if (wid > 0) v += wbuf[wid - 1];
  total = wbuf[kWarps - 1];
  __syncthreads();
  return v;
}

// First index i in [0, n) with a[i] > x (n if none).
__device__ int upper_bound(const int32_t *a, int n, long long x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (a[mid] > x) hi = mid;
    else lo = mid + 1;
  }
  return lo;
}

template <int kPlanThreads>
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const int32_t *__restrict__ lens_in,
                                                            int B, int tile, int C, int kind,
                                                            int splits, int32_t *tm,
                                                            long long s_cap, int staged) {
  // Let the attention kernel that follows start its prologue now; it waits for
  // this grid's completion before it reads the map.
  pdl_launch_dependents();
  // Launched with programmatic serialisation, this grid may start while the kernel
  // before it (the previous step's combine, which reads the map) still runs: read the
  // lengths and write the map only after that grid has completed.
  pdl_wait();
  const TaskMapLayout lay = TaskMapLayout::make(B, C);
  int32_t *lens = tm + lay.lens, *cu_g = tm + lay.cu_tiles, *cb_g = tm + lay.cta_begin;
  int32_t *cs = tm + lay.cta_seg, *so = tm + lay.seg_off;
  int4 *seg = reinterpret_cast<int4 *>(tm + lay.segs);
  // Working copies of cu_tiles and cta_begin: in shared memory when they fit
  // (the binary searches below then cost shared- instead of L2 latency).
  extern __shared__ __align__(8) int32_t stage_buf[];
  int32_t *cu = staged ? stage_buf : cu_g;
  int32_t *cb = staged ? stage_buf + B + 1 : cb_g;
  // keys before each request (token-weighted map only; always staged then)
  long long *kc = reinterpret_cast<long long *>(stage_buf + ((B + 1 + C + 1 + 1) & ~1));
  __shared__ long long wbuf[kPlanThreads / 32];
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  if (tid == 0) s_bad = 0;
  __syncthreads();

  // a1 + a2: tile counts and their running sum (and, for kind 2, the key prefix)
  long long carry = 0, kcarry = 0, total;
  for (int base = 0; base < B; base += kPlanThreads) {
    const int i = base + tid;
    long long n = 0, keys = 0;
    if (i < B) {
      const int L = lens_in[i];
      lens[i] = L;
      if (L < 1) atomicOr(&s_bad, HPA_STATUS_BAD_SEQLEN);
      else n = (L - 1) / tile + 1, keys = L;
    }
    const long long incl = block_scan<kPlanThreads>(n, wbuf, total);
    if (i < B) cu[i + 1] = cu_g[i + 1] = static_cast<int32_t>(carry + incl);
    carry += total;
    if (kind == 2) {
      const long long kincl = block_scan<kPlanThreads>(keys, wbuf, total);
      if (i < B) kc[i + 1] = kcarry + kincl;
      kcarry += total;
    }
  }
  if (tid == 0) {
    cu[0] = cu_g[0] = 0;
    if (kind == 2) kc[0] = 0;
  }
  if (kind == 2 && kcarry > (1ll << 40) && tid == 0) atomicOr(&s_bad, HPA_STATUS_OVERFLOW);
  if (carry > INT_MAX && tid == 0) atomicOr(&s_bad, HPA_STATUS_OVERFLOW);
  __syncthreads();
  const long long T = carry;
  const int bad = s_bad;
  if (bad) {
    if (tid == 0) {
      for (int w = 0; w < TM_HEADER_WORDS; ++w) tm[w] = 0;
      tm[TM_C] = C;
      tm[TM_B] = B;
      tm[TM_TILE] = tile;
      tm[TM_KIND] = kind;
      tm[TM_SPLITS] = splits;
      tm[TM_SCAP] = static_cast<int32_t>(s_cap);
      tm[TM_STATUS] = bad;
    }
    return;
  }

  // a3: partition ranges over the stream
  const long long tbase = T / C, trem = T % C;
  for (int c = tid; c < C; c += kPlanThreads) {
    long long begin;
    if (kind == 0) {
      begin = c * tbase + (c < trem ? c : trem);
    } else if (kind == 2) {
      // first tile whose doubled middle key 2 P_t + w_t reaches X = ceil(2 K c / C)
      const long long K = kcarry;
      const long long X = (2 * K * c + C - 1) / C;
      // last tile of request r has 2 P + w = kc[r] + kc[r+1] + (n_r - 1) * tile
      int lo = 0, hi = B;  // smallest r with that >= X (B if none)
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        const long long e = kc[mid] + kc[mid + 1] + static_cast<long long>(cu[mid + 1] - cu[mid] - 1) * tile;
        if (e >= X) hi = mid;
        else lo = mid + 1;
      }
      if (c == 0) {
        begin = 0;
      } else if (lo == B) {
        begin = T;
      } else {
        const int n = cu[lo + 1] - cu[lo];
        // full tile i: 2 P + w = 2 kc[r] + (2 i + 1) tile >= X  <=>  i >= (X - 2 kc - tile) / (2 tile)
        const long long num = X - 2 * kc[lo] - tile;
        long long i0 = num <= 0 ? 0 : (num + 2 * tile - 1) / (2 * tile);
        if (i0 > n - 1) i0 = n - 1;  // otherwise the last tile (its middle reaches X)
        begin = cu[lo] + i0;
      }
    } else {
      const int r = c / splits, s = c % splits;
      const int n = cu[r + 1] - cu[r];
      const int k = n < splits ? n : splits;
      if (s < k) {
        const int b = n / k, rm = n % k;
        begin = cu[r] + s * b + (s < rm ? s : rm);
      } else {
        begin = cu[r + 1];
      }
    }
    cb[c] = cb_g[c] = static_cast<int32_t>(begin);
  }
  if (tid == 0) cb[C] = cb_g[C] = static_cast<int32_t>(T);
  __syncthreads();

  // a4: segments per partition, their running sum, then the segment rows
  carry = 0;
  int first_rf = 0, first_rl = -1;  // requests of partition tid, kept for the row pass
  for (int base = 0; base < C; base += kPlanThreads) {
    const int c = base + tid;
    long long cnt = 0;
    if (c < C) {
      const int b = cb[c], e = cb[c + 1];
      if (e > b) {
        const int rf = upper_bound(cu, B + 1, b) - 1;
        const int rl = upper_bound(cu, B + 1, e - 1) - 1;
        cnt = rl - rf + 1;
        if (base == 0) first_rf = rf, first_rl = rl;
      }
    }
    const long long incl = block_scan<kPlanThreads>(cnt, wbuf, total);
    if (c < C) cs[c] = static_cast<int32_t>(carry + incl - cnt);
    carry += total;
  }
  const long long S = carry;
  if (tid == 0) cs[C] = static_cast<int32_t>(S);
  if (S > s_cap) {  // cannot happen for maps sized by the library's own queries
    if (tid == 0) tm[TM_STATUS] = HPA_STATUS_OVERFLOW;
    return;
  }
  __syncthreads();
  for (int c = tid; c < C; c += kPlanThreads) {
    const int b = cb[c], e = cb[c + 1];
    if (e <= b) continue;
    const int rf = c == tid ? first_rf : upper_bound(cu, B + 1, b) - 1;
    const int rl = c == tid ? first_rl : upper_bound(cu, B + 1, e - 1) - 1;
    int out = cs[c];
    for (int r = rf; r <= rl; ++r, ++out) {
      const int lo = (b > cu[r] ? b : cu[r]) - cu[r];
      const int hi = (e < cu[r + 1] ? e : cu[r + 1]) - cu[r];
      seg[out] = make_int4(r, lo, hi, c);
      if (lo == 0) so[r] = out;  // the partition holding r's first tile holds its first segment
    }
  }
  for (long long s = S + tid; s < s_cap; s += kPlanThreads) seg[s] = make_int4(-1, -1, -1, -1);
  if (tid == 0) {
    so[B] = static_cast<int32_t>(S);
    for (int w = TM_SCAP + 1; w < TM_HEADER_WORDS; ++w) tm[w] = 0;
    tm[TM_T] = static_cast<int32_t>(T);
    if (kind == 2) {  // key budget: K / C (clamped) and K % C
      const long long kb = kcarry / C;
      tm[TM_BASE] = static_cast<int32_t>(kb > INT_MAX ? INT_MAX : kb);
      tm[TM_REM] = static_cast<int32_t>(kcarry % C);
    } else {
      tm[TM_BASE] = kind == 0 ? static_cast<int32_t>(tbase) : -1;
      tm[TM_REM] = kind == 0 ? static_cast<int32_t>(trem) : -1;
    }
    tm[TM_C] = C;
    tm[TM_B] = B;
    tm[TM_S] = static_cast<int32_t>(S);
    tm[TM_STATUS] = 0;
    tm[TM_TILE] = tile;
    tm[TM_KIND] = kind;
    tm[TM_SPLITS] = splits;
    tm[TM_SCAP] = static_cast<int32_t>(s_cap);
  }
}

}  // namespace

size_t plan_stage_bytes(int B, int C, int kind) {
  size_t words = (static_cast<size_t>(B) + 1 + C + 1 + 1) & ~static_cast<size_t>(1);
  if (kind == 2) words += 2 * (static_cast<size_t>(B) + 1);  // int64 key prefix
  return words * sizeof(int32_t);
}

cudaError_t launch_plan(const int32_t *seq_lens, int B, int tile, int C, int kind, int splits,
                        int32_t *tm, int64_t s_cap, cudaStream_t s) {
  // cu_tiles and cta_begin (and the key prefix) are staged in shared memory when
  // they fit in 40 KB; the token-weighted map requires it (checked by the caller)
  const size_t stage_bytes = plan_stage_bytes(B, C, kind);
  const int staged = stage_bytes <= kPlanStageLimit;
  const size_t smem = staged ? stage_bytes : 0;
  const int need = B > C ? B : C;
  // Programmatic dependent launch: the block's launch overlaps the end of the kernel
  // before it, and pdl_wait() in the kernel orders every read and write after it.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int32_t *lens = seq_lens;
  if (need <= 32) {
    cfg.blockDim = dim3(32);
    return cudaLaunchKernelEx(&cfg, plan_kernel<32>, lens, B, tile, C, kind, splits, tm,
                              static_cast<long long>(s_cap), staged);
  }
  if (need <= 128) {
    cfg.blockDim = dim3(128);
    return cudaLaunchKernelEx(&cfg, plan_kernel<128>, lens, B, tile, C, kind, splits, tm,
                              static_cast<long long>(s_cap), staged);
  }
  if (need <= 256) {
    cfg.blockDim = dim3(256);
    return cudaLaunchKernelEx(&cfg, plan_kernel<256>, lens, B, tile, C, kind, splits, tm,
                              static_cast<long long>(s_cap), staged);
  }
  cfg.blockDim = dim3(1024);
  return cudaLaunchKernelEx(&cfg, plan_kernel<1024>, lens, B, tile, C, kind, splits, tm,
                            static_cast<long long>(s_cap), staged);
}

}  // namespace hpa
