// Fused KV-cache writer: RoPE + RMSNorm + Hadamard + quantisation + paged store,
// one pass ("Hy3 Preview AI Infra 推理优化精读笔记", §4.1 "Rope + Norm + Hadamard +
// Quant + Store KV": the element-wise chain after the QKV projection, fused so
// the new keys and values go from registers straight into the low-bit cache).
//
// Warps walk (token, chunk of 8 KV heads) items, double-buffering each item's
// raw K and V rows in shared memory with asynchronous copies; four KV heads at
// a time (8 lanes per head, 16 dims per lane).  For the key: rotate-half RoPE with the caller's
// cos/sin table, RMSNorm over the 128 dims, optional orthonormal Walsh-Hadamard
// transform, then E4M3 codes of x / scale (round to nearest even, saturating)
// or bf16.  The value is only converted.  Token j of request r is written at
// position L_r - q_len + j.  The arithmetic runs on the packed FP32 pipe: one
// instruction takes two adjacent dims, each rounded as the scalar operation would
// round it (90.3 -> 83.9 us on 65,536 tokens with 8 KV heads).
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


// 16 bf16 (two 16-byte pieces of a row) -> 8 packed fp32 pairs (element 2 j of the
// lane's 16 dims in the low half of x[j]): a bf16 is the high half of
// its fp32, so each word gives its pair with a shift and a mask.
__device__ __forceinline__ void unpack16(const uint4 (&raw)[2], f32x2 (&x)[8]) {
  const uint4 a = raw[0], b = raw[1];
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i)
    x[i] = pk(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}

// scale * x[0..7] -> dims 8k.., scale * x[8..15] -> dims 64 + 8k.. of pool row `row`
// (bf16, or E4M3 codes: round to nearest even, saturating).
__device__ __forceinline__ void store16(void *pool, int kv_dtype, int64_t row, int k,
                                        const f32x2 (&x)[8], float scale) {
  const f32x2 s2 = pk(scale, scale);
  float v[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) upk(mul2(x[i], s2), v[2 * i], v[2 * i + 1]);
  if (kv_dtype == HPA_KV_BF16) {
    __nv_bfloat16 *base = static_cast<__nv_bfloat16 *>(pool) + row * HEAD_DIM;
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = pack_bf16(v[2 * i], v[2 * i + 1]);
    reinterpret_cast<uint4 *>(base + 8 * k)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4 *>(base + 64 + 8 * k)[0] = make_uint4(w[4], w[5], w[6], w[7]);
  } else {
    uint8_t *base = static_cast<uint8_t *>(pool) + row * HEAD_DIM;
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = f32x2_to_e4m3x2(v[4 * i], v[4 * i + 1]);
      const uint32_t hi = f32x2_to_e4m3x2(v[4 * i + 2], v[4 * i + 3]);
      q[i] = lo | (hi << 16);
    }
    reinterpret_cast<uint2 *>(base + 8 * k)[0] = make_uint2(q[0], q[1]);
    reinterpret_cast<uint2 *>(base + 64 + 8 * k)[0] = make_uint2(q[2], q[3]);
  }
}

// RoPE + RMSNorm + (Hadamard) of one key row, 16 dims in this lane (see above).
// The row's scalar factors -- 1 / rms, and 1 / sqrt(128) with the transform -- are
// linear and common to the row, so they are not applied here: y leaves as
// H (w * rope(x)) (or w * rope(x)), and the returned factor is applied once, with the
// cache scale, where the row is stored.
// Packed: y[j] holds dims (2 j, 2 j + 1) of the lane's 16 (j < 4: dims 8k + 2j.., j >= 4:
// 64 + 8k + 2 (j - 4)..); c, sn and w are paired the same way, and nsn = -sn.
__device__ __forceinline__ float key_transform(f32x2 (&y)[8], const f32x2 (&c)[4],
                                               const f32x2 (&sn)[4], const f32x2 (&nsn)[4],
                                               const f32x2 (&w)[8], float eps,
                                               int use_hadamard) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {  // rotate-half RoPE: (y_i, y_{i+64}) turned by angle i
    const f32x2 lo = y[j], hi = y[4 + j];
    y[j] = fma2(hi, nsn[j], mul2(lo, c[j]));
    y[4 + j] = fma2(lo, sn[j], mul2(hi, c[j]));
  }
  f32x2 s2 = mul2(y[0], y[0]);
#pragma unroll
  for (int j = 1; j < 8; ++j) s2 = fma2(y[j], y[j], s2);
  float s0, s1;
  upk(s2, s0, s1);
  float ss = s0 + s1;
  ss += __shfl_xor_sync(kFull, ss, 1);
  ss += __shfl_xor_sync(kFull, ss, 2);
  ss += __shfl_xor_sync(kFull, ss, 4);
  float f = rsqrtf(ss / HEAD_DIM + eps);
#pragma unroll
  for (int j = 0; j < 8; ++j) y[j] = mul2(y[j], w[j]);
  if (!use_hadamard) return f;
  // orthonormal Walsh-Hadamard transform, Sylvester order: a butterfly
  // (a, b) -> (a + b, a - b) over every dim bit.  In registers: dim bit 0 inside a
  // pair, bits 1-2 and 6 between pairs (pair index bits 0-1 and 2)
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float a, b;
    upk(y[j], a, b);
    y[j] = pk(a + b, a - b);
  }
#pragma unroll
  for (int st = 1; st < 8; st <<= 1) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (!(j & st)) {
        const f32x2 a = y[j], b = y[j | st];
        y[j] = add2(a, b);
        y[j | st] = sub2(a, b);
      }
  }
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 1; m < kLanesPerHead; m <<= 1) {  // dim bits 3-5: partner lane ^ m
    // the lane holding a keeps a + b, the one holding b gets a - b: partner + sign * own
    const float sgn = (lane & m) ? -1.f : 1.f;
    const f32x2 sg2 = pk(sgn, sgn);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float a, b;
      upk(y[j], a, b);
      y[j] = fma2(sg2, y[j], pk(__shfl_xor_sync(kFull, a, m), __shfl_xor_sync(kFull, b, m)));
    }
  }
  return f * 0.08838834764831845f;  // 1 / sqrt(128)
}

// 16-byte asynchronous global -> shared copies (cp.async), grouped per token.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_1() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// An item is one new token (r, j) and a chunk of up to 8 of its KV heads; each
// warp keeps two items' raw K and V rows and cos/sin row in its own shared-memory
// slots (4.5 KB each), so the next item's rows stream in while this one's
// arithmetic runs.
constexpr int kChunkHeads = 8;
constexpr int kRowsBytes = kChunkHeads * HEAD_DIM * 2 * 2;  // K then V, bf16
constexpr int kCosOff = kRowsBytes;                         // then the token's cos/sin row
constexpr int kSlotBytes = kRowsBytes + HEAD_DIM * 4;
constexpr int kWarpSmem = 2 * kSlotBytes;

struct Item {
  int64_t rj;  // token index r * q_len + j
  int r, j;    // request and new token within it
  int hc;      // first head of the chunk
  int nh;      // heads in the chunk
};

// A warp's items are it0, it0 + stride, ...: their coordinates advance by fixed
// quotients, so the integer divisions are done once per warp, not per item.
struct ItemWalk {
  int64_t d_rj;  // stride / n_chunks
  int d_ch;      // stride % n_chunks (chunks, 0 .. n_chunks - 1)
  int64_t d_r;   // d_rj / q_len
  int d_j;       // d_rj % q_len
  int n_chunks, q_len, Hkv;

  __device__ Item first(int64_t it) const {
    Item x;
    x.rj = it / n_chunks;
    const int ch = static_cast<int>(it - x.rj * n_chunks);
    x.r = static_cast<int>(x.rj / q_len);
    x.j = static_cast<int>(x.rj - static_cast<int64_t>(x.r) * q_len);
    x.hc = ch * kChunkHeads;
    x.nh = min(kChunkHeads, Hkv - x.hc);
    return x;
  }
  __device__ Item next(const Item &x) const {
    Item y;
    int ch = x.hc / kChunkHeads + d_ch;
    int64_t drj = d_rj;
    if (ch >= n_chunks) ch -= n_chunks, ++drj;  // one carry at most: d_ch < n_chunks
    y.rj = x.rj + drj;
    int j = x.j + d_j + static_cast<int>(drj - d_rj);
    int64_t r = x.r + d_r;
    if (j >= q_len) j -= q_len, ++r;  // d_j + 1 <= q_len, so one carry at most
    y.r = static_cast<int>(r);
    y.j = j;
    y.hc = ch * kChunkHeads;
    y.nh = min(kChunkHeads, Hkv - y.hc);
    return y;
  }
};

// Issue the copies of an item's K and V rows (nh * 256 bytes each) into a slot.
__device__ __forceinline__ void fetch_item(const Item &x, const __nv_bfloat16 *k_new,
                                           const __nv_bfloat16 *v_new, int Hkv, uint32_t slot,
                                           int lane) {
  const int64_t src = (x.rj * Hkv + x.hc) * HEAD_DIM;
  const int chunks = x.nh * (HEAD_DIM * 2 / 16);  // 16-byte chunks per tensor
  const __nv_bfloat16 *ks = k_new + src + 8 * lane, *vs = v_new + src + 8 * lane;
  const uint32_t dk = slot + 16 * lane;
  if (chunks == kChunkHeads * (HEAD_DIM * 2 / 16)) {  // a full chunk: 4 copies per tensor
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      cp_async16(dk + 512 * u, ks + 256 * u);
      cp_async16(dk + kRowsBytes / 2 + 512 * u, vs + 256 * u);
    }
  } else {
    for (int c = lane; c < chunks; c += 32) {
      cp_async16(slot + 16 * c, k_new + src + 8 * c);
      cp_async16(slot + kRowsBytes / 2 + 16 * c, v_new + src + 8 * c);
    }
  }
}

// Where an item's token goes: its position, its page (or -1) and whether both are
// valid; looked up one item ahead, when the item's rows are fetched.
struct Place {
  int pos, page;
  bool good;
};

__device__ __forceinline__ Place look_up(const Item &x, const int32_t *seq_lens,
                                         const int32_t *page_indptr,
                                         const int32_t *page_indices, int64_t num_pages,
                                         int max_pos, int q_len) {
  Place pl;
  const int r = x.r, j = x.j;
  pl.pos = seq_lens[r] - q_len + j;
  pl.page = -1;
  if (pl.pos >= 0 && pl.pos < max_pos) {
    const int pi = page_indptr[r] + pl.pos / PAGE;
    pl.page = pi < page_indptr[r + 1] ? page_indices[pi] : -1;
  }
  pl.good = pl.pos >= 0 && pl.pos < max_pos && pl.page >= 0 && pl.page < num_pages;
  return pl;
}

// The token's cos/sin row (HEAD_DIM floats) into the slot, one 16-byte chunk per lane.
__device__ __forceinline__ void fetch_cos_sin(const Place &pl, const float *cos_sin,
                                              uint32_t slot, int lane) {
  if (pl.good)
    cp_async16(slot + kCosOff + 16 * lane,
               cos_sin + static_cast<int64_t>(pl.pos) * HEAD_DIM + 4 * lane);
}

// Warps walk the items grid-stride; each holds its next item's rows in flight
// (one cp.async group) while it works on the current one.
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
  extern __shared__ __align__(16) uint8_t kv_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int k = lane % kLanesPerHead, hp = lane / kLanesPerHead;
  const uint32_t slots = smem_u32(kv_smem + warp * kWarpSmem);
  const int n_chunks = (Hkv + kChunkHeads - 1) / kChunkHeads;
  const int64_t n_items = static_cast<int64_t>(B) * q_len * n_chunks;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps;
  int64_t it = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  if (it >= n_items) return;

  // RMSNorm weights of this lane's 16 dims (the same for every item)
  f32x2 w[8];
  {
    const float4 *wv = reinterpret_cast<const float4 *>(norm_w);
    const float4 w0 = wv[2 * k], w1 = wv[2 * k + 1], w2 = wv[16 + 2 * k], w3 = wv[16 + 2 * k + 1];
    w[0] = pk(w0.x, w0.y), w[1] = pk(w0.z, w0.w), w[2] = pk(w1.x, w1.y), w[3] = pk(w1.z, w1.w);
    w[4] = pk(w2.x, w2.y), w[5] = pk(w2.z, w2.w), w[6] = pk(w3.x, w3.y), w[7] = pk(w3.z, w3.w);
  }
  const bool e4m3 = kv_dtype == HPA_KV_E4M3;
  // With one chunk of heads (Hkv <= 8) a lane always serves heads hp and 4 + hp: their
  // inverse cache scales are read once
  float rk0[2] = {1.f, 1.f}, rv0[2] = {1.f, 1.f};
  const bool one_chunk = n_chunks == 1;
  if (e4m3 && one_chunk)
#pragma unroll
    for (int ps = 0; ps < 2; ++ps) {
      const int h = ps * kHeadsPerPass + hp;
      if (h < Hkv) rk0[ps] = 1.f / k_scale[h], rv0[ps] = 1.f / v_scale[h];
    }
  ItemWalk walk;
  walk.n_chunks = n_chunks;
  walk.q_len = q_len;
  walk.Hkv = Hkv;
  walk.d_rj = stride / n_chunks;
  walk.d_ch = static_cast<int>(stride - walk.d_rj * n_chunks);
  walk.d_r = walk.d_rj / q_len;
  walk.d_j = static_cast<int>(walk.d_rj - walk.d_r * q_len);
  Item cur = walk.first(it);
  Place here = look_up(cur, seq_lens, page_indptr, page_indices, num_pages, max_pos, q_len);
  fetch_item(cur, k_new, v_new, Hkv, slots, lane);
  fetch_cos_sin(here, cos_sin, slots, lane);
  cp_async_commit();
  for (int buf = 0; it < n_items; it += stride, buf ^= 1) {
    // next item: its rows, its place and its cos/sin row, into the other slot (an
    // empty group when there is none)
    const int64_t nx = it + stride;
    Item nxt = cur;
    Place there = here;
    if (nx < n_items) {
      nxt = walk.next(cur);
      const uint32_t other = slots + (buf ^ 1) * kSlotBytes;
      fetch_item(nxt, k_new, v_new, Hkv, other, lane);
      there = look_up(nxt, seq_lens, page_indptr, page_indices, num_pages, max_pos, q_len);
      fetch_cos_sin(there, cos_sin, other, lane);
    }
    cp_async_commit();

    // the current token: report a bad position or page once per token
    const int pos = here.pos, page = here.page;
    const bool good = here.good;
    if (lane == 0 && status && cur.hc == 0 && !good)
      atomicOr(reinterpret_cast<int *>(status), pos < 0 || pos >= max_pos ? HPA_STATUS_BAD_SEQLEN
                                                                         : HPA_STATUS_BAD_PAGE);
    cp_async_wait_1();  // this item's group has landed (the next one may still fly)
    __syncwarp();
    const uint32_t slot = slots + buf * kSlotBytes;
    if (good) {
      // cos of dims 8k..8k+7 (floats 8k..), sin of the same (floats 64 + 8k..)
      f32x2 c[4], sn[4], nsn[4];
      {
        uint32_t w[16];
        lds128(slot + kCosOff + 32 * k, w[0], w[1], w[2], w[3]);
        lds128(slot + kCosOff + 32 * k + 16, w[4], w[5], w[6], w[7]);
        lds128(slot + kCosOff + 256 + 32 * k, w[8], w[9], w[10], w[11]);
        lds128(slot + kCosOff + 256 + 32 * k + 16, w[12], w[13], w[14], w[15]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          c[j] = pk(__uint_as_float(w[2 * j]), __uint_as_float(w[2 * j + 1]));
          sn[j] = pk(__uint_as_float(w[8 + 2 * j]), __uint_as_float(w[9 + 2 * j]));
          nsn[j] = pk(-__uint_as_float(w[8 + 2 * j]), -__uint_as_float(w[9 + 2 * j]));
        }
      }
#pragma unroll
      for (int ps = 0; ps < kChunkHeads / kHeadsPerPass; ++ps) {
        const int hh = ps * kHeadsPerPass + hp;  // head within the chunk
        const bool active = hh < cur.nh;  // lanes of a missing head still take the shuffles
        f32x2 y[8];
        const uint32_t ka = slot + hh * (HEAD_DIM * 2) + 16 * k;
        if (active) {
          uint4 kr[2];
          lds128(ka, kr[0].x, kr[0].y, kr[0].z, kr[0].w);
          lds128(ka + 128, kr[1].x, kr[1].y, kr[1].z, kr[1].w);
          unpack16(kr, y);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) y[j] = 0ull;
        }
        const float fk = key_transform(y, c, sn, nsn, w, eps, use_hadamard);
        if (active) {
          const int h = cur.hc + hh;
          const int64_t row = (static_cast<int64_t>(page) * Hkv + h) * PAGE + pos % PAGE;
          const float rk = !e4m3 ? 1.f : one_chunk ? rk0[ps] : 1.f / k_scale[h];
          store16(k_pool, kv_dtype, row, k, y, fk * rk);
          // the value, loaded only now: its registers are not live across the key's
          // transform
          uint4 vr[2];
          f32x2 x[8];
          lds128(ka + kRowsBytes / 2, vr[0].x, vr[0].y, vr[0].z, vr[0].w);
          lds128(ka + kRowsBytes / 2 + 128, vr[1].x, vr[1].y, vr[1].z, vr[1].w);
          unpack16(vr, x);
          const float rv = !e4m3 ? 1.f : one_chunk ? rv0[ps] : 1.f / v_scale[h];
          store16(v_pool, kv_dtype, row, k, x, rv);  // value: converted only
        }
      }
    }
    __syncwarp();  // every lane is done with this slot before it is refilled
    cur = nxt;
    here = there;
  }
  cp_async_wait_1();  // nothing of this warp's is left landing in shared memory
}

}  // namespace

cudaError_t launch_store_kv(const StoreKvParams &p, cudaStream_t s) {
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  constexpr int kSmem = kWarps * kWarpSmem;  // 72 KB: two 4.5 KB slots per warp
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(store_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  int sms = 0, per_sm = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, store_kv_kernel, kWarps * 32, kSmem);
  if (e != cudaSuccess) return e;
  // one resident wave of warps that walk the items grid-stride
  const int64_t n_items = static_cast<int64_t>(p.B) * p.q_len *
                          ((p.Hkv + kChunkHeads - 1) / kChunkHeads);
  const int64_t want = (n_items + kWarps - 1) / kWarps;
  const int64_t wave = static_cast<int64_t>(sms) * (per_sm > 0 ? per_sm : 1);
  const unsigned blocks = static_cast<unsigned>(want < wave ? want : wave);
  store_kv_kernel<<<blocks, kWarps * 32, kSmem, s>>>(
      p.k_new, p.v_new, p.seq_lens, p.page_indptr, p.page_indices, p.num_pages, p.cos_sin,
      p.max_pos, p.norm_w, p.eps, p.use_hadamard, p.kv_dtype, p.k_scale, p.v_scale, p.k_pool,
      p.v_pool, p.B, p.q_len, p.Hkv, p.status);
  return cudaGetLastError();
}

}  // namespace hpa
