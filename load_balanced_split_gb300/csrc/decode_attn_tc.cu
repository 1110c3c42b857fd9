// Split-KV GQA decode attention on the 5th-generation tensor cores (tcgen05),
// driven by the same task map and writing the same partials as decode_attn.cu.
//
// "Hy3 Preview AI Infra 推理优化精读笔记", §3.1 方案 steps 4-5: each CTA takes the
// tiles of its partition from the task map and writes split-KV partial
// results for the combine.  One CTA is (partition c, KV head h) and covers all
// G * q_len query rows of h (up to 64) in one pass over the KV, where the
// mma.sync kernel needs one pass per group of 16 rows.  This matters for MTP
// with several draft tokens, where the warp-level MMAs become the bound.
//
// Work per step = PPS pages (64 PPS keys) of one KV head, PPS = 4 for the 8-bit
// path and 2 for bf16; per 128-key tile:
//   S^T[128 keys][rows]  = K[128 keys][128 dims] . Q^T          (tcgen05.mma, TMEM)
//   P^T = 2^(S^T - m)    by the compute threads, one key each    (registers -> smem,
//                        MN-major: each thread stores its key's row with 16-byte stores)
//   O^T[128 dims][rows] += V^T[128 dims][64 PPS keys] . P^T      (tcgen05.mma, TMEM)
// Keys sit on the TMEM lanes for the softmax, so all compute warps share it;
// output dims sit on the lanes for O, so each compute thread owns one dim at
// the segment end and O needs no cross-warp merge.  The row sums l are
// accumulated in fp32 from the unrounded probabilities, per thread (its key
// slot) across the steps, and reduced once per segment.
//
// E4M3 pages feed the MMA as they are (kind::f8f6f4).  The query rows and the
// probabilities are each split into two E4M3 terms, hi = e4m3(x) and
// lo = e4m3(x - hi), side by side in N: their sum carries about 8 significant
// bits, the precision of bf16, so no widening pass is needed.  Queries are
// scaled per row by a power of two into the E4M3 range (folded into the score
// scale), so a bf16 query row is carried exactly.  Probabilities are
// 2^(s - m + 4) with a reference max m that moves only when a score exceeds it
// by more than 4 (base 2), so P <= 256.  bf16 pages use kind::f16 with bf16 Q
// and P.
//
// Roles: CW = 8 or 12 compute warps (softmax, epilogue; the warps with w % 4
// equal share TMEM lane quarter w % 4 -- the same keys, and the same output
// dims -- and split the query rows, 8, 16 or 32 rows each), then one TMA
// producer warp, one warp whose thread issues Q K^T and one issuing P V.  A
// tcgen05.mma costs its issuing thread about 100 cycles whatever N is, so the
// two products are issued from two threads and each step issues few, wide
// MMAs.  S is double-buffered in TMEM (single-buffered at 64 E4M3 rows) so Q K^T
// of step i+1 overlaps the softmax of step i.  Every wait is
// bounded in time; a role that gives up flags the task map's status word and
// raises the CTA's abort flag, each MMA thread commits its MMAs to a drain
// barrier that the CTA waits on, the producer waits for its copies, and the
// CTA frees its TMEM and returns.
#include <math_constants.h>

#include <climits>

#include "hpa_internal.cuh"

namespace hpa {
namespace {

constexpr uint32_t kFull = 0xffffffffu;

template <int KV>
struct TcCfg;
template <>
struct TcCfg<HPA_KV_BF16> {
  static constexpr int kPageBytes = 16384;  // one page-head of K (or V)
  static constexpr float kSlack = 8.f;      // P <= 2^8 in bf16
  static constexpr float kPOff = 0.f;
};
template <>
struct TcCfg<HPA_KV_E4M3> {
  static constexpr int kPageBytes = 8192;
  static constexpr float kSlack = 4.f;      // P = 2^(s - m + 4) <= 2^8 = 256 < 448
  static constexpr float kPOff = 4.f;
};

// Shared memory of one CTA; NC = row chunks of 16 (Rp = 16 NC padded rows).
template <int KV, int NC>
struct TcSmem {
  static constexpr int kRp = 16 * NC;
  // Compute warps: 4 per group of rows, one group per TMEM lane quarter each (8
  // warps up to 32 rows, 12 for 48 and 8 of 32 rows each for 64).  At 64 rows, 16
  // warps of 16 rows would leave 96 registers a thread (19 warps, 5 on some SM
  // sub-partitions); 8 warps of 32 rows get 168 (11 warps) and were 1.2 % faster.
  static constexpr int kCW = NC <= 2 || NC == 4 ? 8 : 4 * NC;
  static constexpr int kRH = kRp / (kCW / 4);                  // rows per compute warp
  static constexpr int kThreads = (kCW + 3) * 32;              // + producer, QK, PV issuers
  // Columns of S and of O: the hi and lo terms of the 8-bit path sit side by side
  // (one MMA with N = 2 Rp instead of two with N = Rp: MMA issue, not tensor math,
  // is what a step of narrow MMAs costs).
  static constexpr int kNS = KV == HPA_KV_E4M3 ? 2 * kRp : kRp;
  // Pages per step: every step pays a fixed chain of waits (S ready, the reference-max
  // vote, P V done), so the 8-bit path takes four pages (1790 -> 1449 us at q_len 6,
  // 2093 -> 2040 at q_len 8, against two-page steps).  bf16 stages of four pages would
  // not fit twice in shared memory.
  static constexpr int kPPS = KV == HPA_KV_E4M3 ? 4 : 2;
  // S buffers in TMEM: two (48 rows: 2 x 2 tiles x 96 columns of S + 96 of O = 480 of
  // 512), except at 64 E4M3 rows, where two tiles of 128 columns plus O leave room for
  // one.  With one, Q K^T of step i + 1 waits until step i's scores are in registers
  // and its reference vote is done, and runs under step i's P encoding.
  static constexpr int kSBufs = KV == HPA_KV_E4M3 && NC == 4 ? 1 : 2;
  static constexpr int kMT = kPPS / 2;                         // 128-key tiles per step
  static constexpr int kStepKeys = PAGE * kPPS;
  static constexpr int kKStep = kPPS * TcCfg<KV>::kPageBytes;  // K of one step
  static constexpr int kStageBytes = 2 * kKStep;               // K then V
  static constexpr int kOperand = 256 * kRp;                   // a Q slot
  // P^T is stored MN-major: one row of 2 Rp bytes per key (E4M3: the hi rows, then
  // the lo rows; bf16: the rows), padded to a swizzle width of 32, 64 or 128 bytes.
  // A compute thread owns one key, so it writes its probabilities with vector
  // stores and no exchange between lanes.
  static constexpr int kPSW = NC == 1 ? 32 : NC == 2 ? 64 : 128;  // bytes per key row
  static constexpr int kPSwz = kPSW == 32 ? 6 : kPSW == 64 ? 4 : 2;  // descriptor mode
  static constexpr int kPBuf = kStepKeys * kPSW;
  // P^T of a step is written over the K half of that step's own stage: Q K^T has
  // read K by then (its completion is what the compute warps wait for), and the
  // P V that reads P^T is what releases the stage.  So P^T needs no buffers of
  // its own and the room goes to one more stage.
  static_assert(kPBuf <= kKStep, "P^T fits in the K half of a stage");
  // Up to 32 rows, as many stages as fit beside the operands (one CTA per SM):
  // there DRAM latency is hidden by the bytes in flight (2 -> 3 stages at 32 rows:
  // 1.21x).  With 48 or 64 rows the compute warps are the bound and deeper rings
  // were slower (6 and 5 stages against 4: 5 % and 10 %), so they keep 4.
  static constexpr int kStages0 = (226 * 1024 - 2 * kOperand - 6 * 1024) / kStageBytes;
  static constexpr int kStageCap = NC <= 2 ? 6 : 4;
  static constexpr int kStages = kStages0 > kStageCap ? kStageCap : kStages0;
  static constexpr int kQ = kStages * kStageBytes;             // 2 query slots
  static constexpr int kRowC = kQ + 2 * kOperand;              // float[2][64] score scales
  static constexpr int kStepMax = kRowC + 2 * 64 * 4;          // float[2][4][64]
  static constexpr int kFlags = kStepMax + 2 * 4 * 64 * 4;     // int[2][16]
  static constexpr int kLRed = kFlags + 128;                   // float[4][64] row-sum parts
  static constexpr int kJRow = kLRed + 4 * 64 * 4;             // int[64]: token j of row r
  // From 48 rows on the compute role is short of registers (at 48 rows the two-tile
  // steps, at 64 the 32 rows a warp), so there the per-row biases live in shared
  // memory (one slot of kRH floats per compute warp, read with broadcast loads);
  // below, in registers.
  static constexpr bool kBiasInSmem = NC >= 3;
  static constexpr int kBias = kJRow + 64 * 4;                 // float[kCW][kRH]
  static_assert(kCW * kRH <= 256, "bias slots");
  static constexpr int kInfo = kBias + 16 * 16 * 4;            // int4[2]
  static constexpr int kBars = kInfo + 32;
  // q_full[2] q_empty[2] s_full[2] s_free[2] p_full[2] pv_done[2] o_free drain flag[2]
  // smax lred kv_full[kStages] kv_empty[kStages]
  static constexpr int kNumBars = 30 + 2 * kStages;
  static constexpr int kKvEmpty = 30 + kStages;  // first kv_empty barrier (after kv_full)
  static constexpr int kTmem = kBars + kNumBars * 8;           // TMEM base address
  static constexpr int kAbort = kTmem + 4;
  static constexpr int kBytes = kAbort + 4;
  static constexpr int kAlloc = kBytes + 1024;                 // room to align the base
  static_assert(kAlloc <= 232448, "dynamic shared memory of one CTA");
  // TMEM columns: S[0], S[1] (kMT tiles of kNS each), O (kNS), rounded up to a power
  // of two >= 32
  static constexpr int kCols = (kSBufs * kMT + 1) * kNS;
  static constexpr int kTmemCols =
      kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128 : kCols <= 256 ? 256 : 512;
  static constexpr int kOCol = kSBufs * kMT * kNS;  // first column of O
  static_assert(kCols <= 512, "TMEM");
  static_assert(kStages >= 2, "shared memory");
};

enum TcBar : int {
  B_Q_FULL = 0, B_Q_EMPTY = 2, B_S_FULL = 4, B_S_FREE = 6, B_P_FULL = 8, B_PV_DONE = 10,
  // per row group g (the 4 warps that share rows): flag[b][g], smax[g], lred[g]
  B_O_FREE = 12, B_DRAIN = 13, B_FLAG = 14, B_SMAX = 22, B_LRED = 26, B_KV_FULL = 30
};


// ---- tcgen05 wrappers ---------------------------------------------------------------
// Shared-memory matrix descriptor (sm_100 family): start, leading and stride byte
// offsets in 16-byte units, version 1, swizzle mode (2 = 128-byte, 4 = 64-byte,
// 6 = 32-byte).
__device__ __forceinline__ uint64_t tc_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                            uint32_t swz = 2) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
         (static_cast<uint64_t>(swz) << 61);
}

// Instruction descriptor: fp32 accumulate, M = 128, N = n; A/B formats (bf16 = 1 for
// kind::f16, E4M3 = 0 for kind::f8f6f4) and major-ness (0 = K-major, 1 = MN-major).
__device__ __forceinline__ uint32_t tc_idesc(int fmt, int n, int a_mn, int b_mn) {
  return (1u << 4) | (static_cast<uint32_t>(fmt) << 7) | (static_cast<uint32_t>(fmt) << 10) |
         (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
}

template <int KV>
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  if (KV == HPA_KV_BF16)
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// Arrive on `bar` once every MMA this thread has issued so far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 8 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tc_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tc_st8(uint32_t taddr, const float (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
               "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
               : "memory");
}

__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Two f16 (element 0 in the low half) -> two E4M3 codes, round to nearest even,
// saturating.
__device__ __forceinline__ uint16_t f16x2_to_e4m3x2(uint32_t v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(v));
  return r;
}

__device__ __forceinline__ void sts64(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// 2^k with a * 2^k in [128, 256) for a > 0 (1 for a == 0), k clamped to keep it an
// fp32 normal.
__device__ __forceinline__ float pow2_to_128(float a) {
  int ea = static_cast<int>((__float_as_uint(a) >> 23) & 0xffu) - 127;
  ea = min(max(ea, -119), 126);
  return a > 0.f ? __uint_as_float(static_cast<uint32_t>(127 + 7 - ea) << 23) : 1.f;
}

__device__ __forceinline__ float warp_max(float x) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}

// Byte offset of byte n of key k's row in an MN-major operand whose rows are one
// swizzle width sw (32, 64 or 128 bytes) long, from a 1024-byte aligned base: the
// 16-byte chunk index XOR address bits 7.. (as many bits as the row has chunks - 1).
__device__ __forceinline__ uint32_t mnmaj(int k, int n, int sw) {
  const uint32_t row = static_cast<uint32_t>(k) * sw;
  return row + ((((n >> 4) ^ (row >> 7)) & (sw / 16 - 1)) << 4) + (n & 15);
}

// Byte offset of (row r, byte kb) in a K-major operand with 128-byte swizzle:
// 8-row atoms of 8 x 128 B, 16-byte chunk index XOR (row % 8).  Rows beyond the
// first 128-byte column block live in the next block, `blk` bytes further on.
__device__ __forceinline__ uint32_t kmaj(int r, int kb, uint32_t blk) {
  return (kb >> 7) * blk + (r >> 3) * 1024 + (r & 7) * 128 + ((((kb & 127) >> 4) ^ (r & 7)) << 4) +
         (kb & 15);
}

// ----------------------------------------------------------------------------- roles
template <int KV, int NC>
struct Tc {
  using S = TcSmem<KV, NC>;
  static constexpr int kRp = S::kRp;

  // ---- the TMA warp (after the compute warps): query staging and the K/V copies
  static __device__ void producer(const AttnParams &p, const CUtensorMap *tmk,
                                  const CUtensorMap *tmv, uint8_t *smem, int s_begin,
                                  int s_end, int tile, int h) {
    const int lane = threadIdx.x & 31;
    const uint32_t base = smem_u32(smem), bars = base + S::kBars;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kAbort);
    uint64_t pol = 0;
    if (lane == 0) {
      pol = l2_policy_evict_first();
      prefetch_tmap(tmk);
      prefetch_tmap(tmv);
    }
    const int G = p.G, R = p.rows;
    float ksc = 1.f;
    if (KV == HPA_KV_E4M3) ksc = p.k_scale[h];
    int st = 0;
    uint32_t phase = 0, issued = 0, parity_bits = 0;
    bool ok = true;
    for (int s = s_begin; s < s_end && ok; ++s) {
      const int k = s - s_begin, slot = k & 1;
      const SegRow sr = read_seg_row(p.tm, p.lay, p.B, s, blockIdx.x, tile, lane == 0);
      const int r = sr.r, L = sr.L, klo = sr.klo, khi = sr.khi;
      const int pg0 = klo / PAGE, pg1 = (khi + PAGE - 1) / PAGE;
      int good = 1;
      if (lane == 0)
        good = !*abort_flag && mbar_wait_bounded_rolled(bars + 8 * (B_Q_EMPTY + slot), ((k >> 1) & 1) ^ 1);
      if (!__shfl_sync(kFull, good, 0)) {
        ok = false;
        break;
      }
      // query rows -> operand slot (K-major, 128-byte swizzle); lane l holds dims 4l..4l+3.
      // The rows' loads go out 8 at a time: with one at a time, staging 64 rows took
      // about 28 us of load latency per segment, during which this warp issued no K/V
      // copies and the compute warps drained the ring (measured per CTA against its
      // segment count: 28 -> 10 us per segment at 64 rows, 15 -> 7 at 32).
      uint8_t *qs = smem + S::kQ + slot * S::kOperand;
      float *rowc = reinterpret_cast<float *>(smem + S::kRowC) + slot * 64;
      const int *jrow = reinterpret_cast<const int *>(smem + S::kJRow);
      constexpr int kQB = 8;  // rows whose loads are in flight together
      for (int rb = 0; rb < kRp; rb += kQB) {
        uint2 raws[kQB];
#pragma unroll
        for (int u = 0; u < kQB; ++u) {
          const int row = rb + u;
          raws[u] = make_uint2(0u, 0u);
          if (row < R) {
            const int j = jrow[row], g = row - j * G;
            raws[u] = reinterpret_cast<const uint2 *>(
                p.q + ((static_cast<int64_t>(r) * p.q_len + j) * p.Hq + h * G + g) * HEAD_DIM)[lane];
          }
        }
#pragma unroll
        for (int u = 0; u < kQB; ++u) {
          const int row = rb + u;
          float x[4];
          {
            const uint2 raw = raws[u];
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.x));
            const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.y));
            x[0] = a.x, x[1] = a.y, x[2] = b.x, x[3] = b.y;
          }
          if (KV == HPA_KV_BF16) {
            uint2 w;
            w.x = pack_bf16(x[0], x[1]);
            w.y = pack_bf16(x[2], x[3]);
            *reinterpret_cast<uint2 *>(qs + kmaj(row, 8 * lane, kRp * 128)) = w;
            if (lane == 0) rowc[row] = p.scale_log2;
          } else {
            float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
            amax = warp_max(amax);
            // A power-of-two row scale puts amax * sq in [128, 256) (hi = e4m3 of it).  Every
            // residual x * sq - hi is then at most half an E4M3 step of [128, 256), i.e. 8, so
            // lo = e4m3(16 (x * sq - hi)) never saturates, and hi + lo / 16 carries a bf16
            // element to its 8 significant bits down to 2^-12 of the row's largest (without
            // the 16, residuals of small elements fall under E4M3's smallest step).
            const float sq = pow2_to_128(amax);
            uint32_t hi = 0, lo = 0;
            float res[4];
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
              const float v0 = x[e] * sq, v1 = x[e + 1] * sq;
              const uint16_t h2 = f32x2_to_e4m3x2(v0, v1);
              const uint32_t hh = e4m3x2_to_f16x2(h2);
              const float2 hf = __half22float2(*reinterpret_cast<const __half2 *>(&hh));
              res[e] = v0 - hf.x;  // exact: both have at most 8 significant bits
              res[e + 1] = v1 - hf.y;
              hi |= static_cast<uint32_t>(h2) << (8 * e);
            }
#pragma unroll
            for (int e = 0; e < 4; e += 2)
              lo |= static_cast<uint32_t>(f32x2_to_e4m3x2(16.f * res[e], 16.f * res[e + 1])) << (8 * e);
            *reinterpret_cast<uint32_t *>(qs + kmaj(row, 4 * lane, 0)) = hi;
            *reinterpret_cast<uint32_t *>(qs + kRp * 128 + kmaj(row, 4 * lane, 0)) = lo;
            if (lane == 0) rowc[row] = p.scale_log2 * ksc / sq;
          }
        }
      }
      if (lane == 0)
        reinterpret_cast<int4 *>(smem + S::kInfo)[slot] = make_int4(r, L, klo, khi);
      fence_proxy_async_smem();  // the MMA reads the slot through the async proxy
      mbar_arrive(bars + 8 * (B_Q_FULL + slot));

      // KV pages, kPPS per stage
      constexpr int PPS = S::kPPS;
      const int pstart = p.page_indptr[r];
      const int pcount = p.page_indptr[r + 1] - pstart;
      const int32_t *pidx = p.page_indices + pstart;
      for (int pb = pg0; pb < pg1 && ok; pb += 32 * PPS) {
        int id[PPS];
#pragma unroll
        for (int u = 0; u < PPS; ++u) {
          const int pg = pb + PPS * lane + u;
          id[u] = 0;
          if (pg < pg1) {
            id[u] = pg < pcount ? pidx[pg] : -1;
            if (id[u] < 0 || id[u] >= p.num_pages) {
              status_or(p.tm, HPA_STATUS_BAD_PAGE);
              id[u] = 0;
            }
          }
        }
        const int nstep = min(32, (pg1 - pb + PPS - 1) / PPS);
        for (int i = 0; i < nstep; ++i) {
          const int n = min(PPS, pg1 - (pb + PPS * i));
          int ids[PPS];
#pragma unroll
          for (int u = 0; u < PPS; ++u) ids[u] = __shfl_sync(kFull, id[u], i);
          int g2 = 1;
          if (lane == 0) {
            if (*abort_flag ||
                !mbar_wait_bounded_rolled(bars + 8 * (S::kKvEmpty + st), phase ^ 1)) {
              g2 = 0;
            } else {
              const uint32_t fb = bars + 8 * (B_KV_FULL + st);
              const uint32_t dst = base + st * S::kStageBytes;
              mbar_arrive_expect_tx(fb, n * 2 * TcCfg<KV>::kPageBytes);
#pragma unroll
              for (int u = 0; u < PPS; ++u) {
                if (u >= n) break;
                const int z = ids[u] * p.Hkv + h;
                if (KV == HPA_KV_BF16) {
                  // [dim block][64 PPS keys][128 B] for K, then the same for V
                  constexpr int blk = PPS * 8192;
                  tma_load_3d(dst + u * 8192, tmk, fb, 0, 0, z, pol);
                  tma_load_3d(dst + blk + u * 8192, tmk, fb, 64, 0, z, pol);
                  tma_load_3d(dst + S::kKStep + u * 8192, tmv, fb, 0, 0, z, pol);
                  tma_load_3d(dst + S::kKStep + blk + u * 8192, tmv, fb, 64, 0, z, pol);
                } else {
                  tma_load_3d(dst + u * 8192, tmk, fb, 0, 0, z, pol);
                  tma_load_3d(dst + S::kKStep + u * 8192, tmv, fb, 0, 0, z, pol);
                }
              }
              issued |= 1u << st;
              parity_bits = (parity_bits & ~(1u << st)) | (phase << st);
            }
          }
          ok = __shfl_sync(kFull, g2, 0) != 0;
          if (!ok) break;
          if (++st == S::kStages) {
            st = 0;
            phase ^= 1;
          }
        }
      }
    }
    if (!ok && lane == 0) {
      status_or(p.tm, HPA_STATUS_TIMEOUT);
      *abort_flag = 1;
      for (int i = 0; i < S::kStages; ++i)  // never leave copies landing in shared memory
        if (issued & (1u << i))
          mbar_wait_bounded_rolled(bars + 8 * (B_KV_FULL + i), (parity_bits >> i) & 1u, 1000000000ull);
    }
  }

  // ---- the two MMA warps, one thread each.  Both walk the same segments
  // and steps as the producer; st / i / phase follow the same sequence.
  static __device__ void mma_done(const AttnParams &p, uint8_t *smem, bool ok) {
    const uint32_t bars = smem_u32(smem) + S::kBars;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kAbort);
    if (!ok) {
      status_or(p.tm, HPA_STATUS_TIMEOUT);
      *abort_flag = 1;
    }
    // every MMA this thread issued completes before the CTA frees its TMEM
    tc_commit(bars + 8 * B_DRAIN);
  }

  static __device__ void qk_issuer(const AttnParams &p, uint8_t *smem, int s_begin, int s_end,
                                   int tile, uint32_t tmem) {
    const uint32_t base = smem_u32(smem), bars = base + S::kBars;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kAbort);
    int i = 0, st = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int s = s_begin; s < s_end && ok; ++s) {
      const int k = s - s_begin, slot = k & 1;
      const SegRow sr = read_seg_row(p.tm, p.lay, p.B, s, blockIdx.x, tile, false);
      const int pg0 = sr.klo / PAGE, pg1 = (sr.khi + PAGE - 1) / PAGE;
      const int nsteps = (pg1 - pg0 + S::kPPS - 1) / S::kPPS;
      if (*abort_flag || !mbar_wait_bounded_rolled(bars + 8 * (B_Q_FULL + slot), (k >> 1) & 1)) {
        ok = false;
        break;
      }
      const uint32_t qbase = base + S::kQ + slot * S::kOperand;
      for (int j = 0; j < nsteps; ++j) {
        const int b = i & 1;
        if (*abort_flag || !mbar_wait_bounded_rolled(bars + 8 * (B_KV_FULL + st), phase) ||
            !(S::kSBufs == 2
                  ? mbar_wait_bounded_rolled(bars + 8 * (B_S_FREE + b), ((i >> 1) & 1) ^ 1)
                  // one buffer: step i - 1 must have released it (for i = 0, the barrier
                  // of step -1 passes at once)
                  : mbar_wait_bounded_rolled(bars + 8 * (B_S_FREE + ((i - 1) & 1)), ((i - 1) >> 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kbase = base + st * S::kStageBytes;
#pragma unroll
        for (int mt = 0; mt < S::kMT; ++mt) {  // keys [128 mt, 128 mt + 128) of the step
          const uint32_t s_t = tmem + ((S::kSBufs == 2 ? b : 0) * S::kMT + mt) * S::kNS;
          if (KV == HPA_KV_BF16) {
            const uint32_t id = tc_idesc(1, kRp, 0, 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // 16 dims per MMA
              tc_mma<KV>(s_t,
                         tc_desc(kbase + (kk >> 2) * (S::kPPS * 8192) + mt * 16384 + (kk & 3) * 32,
                                 16, 1024),
                         tc_desc(qbase + (kk >> 2) * (kRp * 128) + (kk & 3) * 32, 16, 1024), id,
                         kk > 0);
          } else {
            // B = [Q hi rows; Q lo rows] (2 Rp rows): S hi in columns [0, Rp), lo in [Rp, 2 Rp)
            const uint32_t id = tc_idesc(0, 2 * kRp, 0, 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // 32 dims per MMA
              tc_mma<KV>(s_t, tc_desc(kbase + mt * 16384 + kk * 32, 16, 1024),
                         tc_desc(qbase + kk * 32, 16, 1024), id, kk > 0);
          }
        }
        tc_commit(bars + 8 * (B_S_FULL + b));
        if (j == nsteps - 1) tc_commit(bars + 8 * (B_Q_EMPTY + slot));
        ++i;
        if (++st == S::kStages) {
          st = 0;
          phase ^= 1;
        }
      }
    }
    mma_done(p, smem, ok);
  }

  static __device__ void pv_issuer(const AttnParams &p, uint8_t *smem, int s_begin, int s_end,
                                   int tile, uint32_t tmem) {
    const uint32_t base = smem_u32(smem), bars = base + S::kBars;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kAbort);
    const uint32_t o_t = tmem + S::kOCol;
    int i = 0, st = 0;
    bool ok = true;
    for (int s = s_begin; s < s_end && ok; ++s) {
      const int k = s - s_begin;
      const SegRow sr = read_seg_row(p.tm, p.lay, p.B, s, blockIdx.x, tile, false);
      const int pg0 = sr.klo / PAGE, pg1 = (sr.khi + PAGE - 1) / PAGE;
      const int nsteps = (pg1 - pg0 + S::kPPS - 1) / S::kPPS;
      for (int j = 0; j < nsteps; ++j) {
        const int b = i & 1;
        // P of this step written; at a segment start, the previous segment's O read out
        if (*abort_flag || !mbar_wait_bounded_rolled(bars + 8 * (B_P_FULL + b), (i >> 1) & 1) ||
            (j == 0 && k > 0 && !mbar_wait_bounded_rolled(bars + 8 * B_O_FREE, (k - 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t vbase = base + st * S::kStageBytes + S::kKStep;
        const uint32_t pbase = base + st * S::kStageBytes;  // P^T over the stage's K
        // A = V^T and B = P^T, both MN-major; B's stride between groups of 8 keys is
        // 8 key rows
        if (KV == HPA_KV_BF16) {
          const uint32_t idv = tc_idesc(1, kRp, 1, 1);
#pragma unroll
          for (int kk = 0; kk < 4 * S::kPPS; ++kk)  // 16 keys per MMA
            tc_mma<KV>(o_t, tc_desc(vbase + kk * 2048, S::kPPS * 8192, 1024),
                       tc_desc(pbase + kk * 16 * S::kPSW, 16, 8 * S::kPSW, S::kPSwz), idv,
                       j > 0 || kk > 0);
        } else {
          // B = [P hi rows; P lo rows]: O hi in columns [0, Rp), lo in [Rp, 2 Rp)
          const uint32_t idv = tc_idesc(0, 2 * kRp, 1, 1);
#pragma unroll
          for (int kk = 0; kk < 2 * S::kPPS; ++kk)  // 32 keys per MMA
            tc_mma<KV>(o_t, tc_desc(vbase + kk * 4096, 8192, 1024),
                       tc_desc(pbase + kk * 32 * S::kPSW, 16, 8 * S::kPSW, S::kPSwz), idv,
                       j > 0 || kk > 0);
        }
        // Q K^T of this step completed before its P was written, so this commit
        // frees the whole K/V stage
        tc_commit(bars + 8 * (S::kKvEmpty + st));
        tc_commit(bars + 8 * (B_PV_DONE + b));  // P[b] is free; O is current
        ++i;
        if (++st == S::kStages) st = 0;
      }
    }
    mma_done(p, smem, ok);
  }

  // ---- the compute warps: softmax and the segment epilogue.  Thread t: key slots
  // kt + 128 m of the step (m < kMT) and output dim kt = t % 128 (its TMEM lane),
  // rows [hf RH, hf RH + RH) with hf = t / 128.
  static __device__ void compute(const AttnParams &p, uint8_t *smem, int s_begin, int s_end,
                                 uint32_t tmem, int h) {
    constexpr int RH = S::kRH;  // rows per warp
    constexpr int MT = S::kMT;
    const int t = threadIdx.x, w = t >> 5, lane = t & 31, qd = w & 3, hf = w >> 2;
    const int kt = t & 127, r0 = hf * RH;  // hf: this warp's group of rows
    const uint32_t base = smem_u32(smem), bars = base + S::kBars;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kAbort);
    const uint32_t lane_t = tmem + (static_cast<uint32_t>(32 * qd) << 16);
    const int G = p.G, R = p.rows, q_len = p.q_len;
    const float vsc = KV == HPA_KV_E4M3 ? p.v_scale[h] : 1.f;
    constexpr float kSlack = TcCfg<KV>::kSlack, kPOff = TcCfg<KV>::kPOff;
    float *stepmax = reinterpret_cast<float *>(smem + S::kStepMax);  // [2][4 quarters][64]
    int *flags = reinterpret_cast<int *>(smem + S::kFlags);           // [2][8 warps]
    float *lred = reinterpret_cast<float *>(smem + S::kLRed);         // [4 quarters][64]
    const int *jrow = reinterpret_cast<const int *>(smem + S::kJRow);
    int i = 0, n_moved = 0, n_seg = 0;
    bool ok = true;
    for (int s = s_begin; s < s_end && ok; ++s) {
      const int k = s - s_begin, slot = k & 1;
      if (*abort_flag || !mbar_wait_bounded_rolled(bars + 8 * (B_Q_FULL + slot), (k >> 1) & 1)) {
        ok = false;
        break;
      }
      const int4 inf = reinterpret_cast<const int4 *>(smem + S::kInfo)[slot];
      const int L = inf.y, klo = inf.z, khi = inf.w;
      const int pg0 = klo / PAGE, pg1 = (khi + PAGE - 1) / PAGE;
      const int nsteps = (pg1 - pg0 + S::kPPS - 1) / S::kPPS;
      if (L < q_len && t == 0) status_or(p.tm, HPA_STATUS_BAD_SEQLEN);
      const uint32_t rowc_s = base + S::kRowC + (slot * 64 + r0) * 4;
      const float c_all = p.scale_log2;  // bf16: one score scale for every row
      // Per row: bo = (reference max) - kPOff, -inf until the row has a reference, and
      // this key slot's share of l.  A probability is 2^(x - bo), x = c * S the score in
      // base 2, so one FMA per element gives the exp2 argument a = c * S - bo.  The
      // biases are kept negated (nb = -bo), the FMA's addend.
      float bo_r[S::kBiasInSmem ? 1 : RH], lsum[RH];
      float *const bo_s = reinterpret_cast<float *>(smem + S::kBias) + w * RH;  // this warp's slot
      // nb of rows e4 .. e4 + 3 of this warp
      auto nbias4 = [&](int e4, float (&v)[4]) {
        if constexpr (S::kBiasInSmem) {
          uint32_t w0, w1, w2, w3;
          lds128(smem_u32(bo_s + e4), w0, w1, w2, w3);
          v[0] = __uint_as_float(w0), v[1] = __uint_as_float(w1);
          v[2] = __uint_as_float(w2), v[3] = __uint_as_float(w3);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) v[e] = bo_r[e4 + e];
        }
      };
      auto bias4 = [&](int e4, float (&v)[4]) {  // bo
        nbias4(e4, v);
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = -v[e];
      };
      auto bias_set = [&](int e, float v) {  // bo; every lane holds the same v
        if constexpr (S::kBiasInSmem) {
          if (lane == 0) bo_s[e] = -v;
        } else {
          bo_r[e] = -v;
        }
      };
      // A row with no reference yet has bias 0 (its a is the plain score x) and its bit set
      // in `unref`; padding rows never get one and have no bit.
#pragma unroll
      for (int e = 0; e < RH; ++e) {
        bias_set(e, 0.f);
        lsum[e] = 0.f;
      }
      uint32_t unref = 0;
#pragma unroll
      for (int e = 0; e < RH; ++e) unref |= (r0 + e < R ? 1u : 0u) << e;
      if constexpr (S::kBiasInSmem) __syncwarp();
      const bool full = r0 + RH <= R;  // every row of this warp is a query row (warp-uniform)

      for (int jp = 0; jp < nsteps; ++jp) {
        const int b = i & 1, st = i % S::kStages;
        if (*abort_flag || !mbar_wait_bounded_rolled(bars + 8 * (B_S_FULL + b), (i >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int key0 = (pg0 + S::kPPS * jp) * PAGE + kt;  // key of slot m: key0 + 128 m
        int d0[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const bool present = key0 + 128 * m < pg1 * PAGE;  // the step's last pages may be missing
          // row r (token j = r / G) sees keys < L - q_len + 1 + j
          d0[m] = present ? key0 + 128 * m - (L - q_len + 1) : INT_MAX;
        }
        // a[m][e] = c_e * S - bo_e for this key slot and the warp's rows: -inf for keys a
        // row may not see and for padding rows.
        float a[MT][RH];
        auto scores = [&]() {
          // The loaded registers are read only after tcgen05.wait::ld: a tile's hi terms
          // land in a, its lo terms (E4M3) in u, and S = S(Q hi) + S(Q lo) / 16 (the lo
          // term's fixed scale) is formed after the wait.
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            float u[KV == HPA_KV_E4M3 ? RH : 1];
#pragma unroll
            for (int c = 0; c < RH / 8; ++c) {
              const uint32_t col = lane_t + ((S::kSBufs == 2 ? b : 0) * MT + m) * S::kNS + r0 + 8 * c;
              tc_ld8(col, *reinterpret_cast<float(*)[8]>(&a[m][8 * c]));
              if (KV == HPA_KV_E4M3) tc_ld8(col + kRp, *reinterpret_cast<float(*)[8]>(&u[8 * c]));
            }
            if (KV == HPA_KV_E4M3) {
              tc_wait_ld();
              const f32x2 k16 = pk(0.0625f, 0.0625f);
#pragma unroll
              for (int e = 0; e < RH; e += 2)
                upk(fma2(pk(u[e], u[e + 1]), k16, pk(a[m][e], a[m][e + 1])), a[m][e], a[m][e + 1]);
            }
          }
          tc_wait_ld();
#pragma unroll
          for (int e4 = 0; e4 < RH; e4 += 4) {
            float c4[4] = {c_all, c_all, c_all, c_all};
            if (KV == HPA_KV_E4M3) {  // per-row scale (the query rows' own power of two)
              uint32_t w0, w1, w2, w3;
              lds128(rowc_s + 4 * e4, w0, w1, w2, w3);
              c4[0] = __uint_as_float(w0), c4[1] = __uint_as_float(w1);
              c4[2] = __uint_as_float(w2), c4[3] = __uint_as_float(w3);
            }
            float nb4[4];
            nbias4(e4, nb4);
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
              for (int e = 0; e < 4; e += 2) {
                const f32x2 s2 = pk(a[m][e4 + e], a[m][e4 + e + 1]), c2 = pk(c4[e], c4[e + 1]);
                upk(fma2(s2, c2, pk(nb4[e], nb4[e + 1])), a[m][e4 + e], a[m][e4 + e + 1]);
              }
          }
          if (!full) {
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
              for (int e = 0; e < RH; ++e)
                if (r0 + e >= R) a[m][e] = -CUDART_INF_F;
          }
#pragma unroll
          for (int m = 0; m < MT; ++m)
            if (__any_sync(kFull, d0[m] >= 0)) {  // near the request's end, or a missing page
#pragma unroll
              for (int e = 0; e < RH; ++e)
                if (d0[m] >= jrow[r0 + e]) a[m][e] = -CUDART_INF_F;
            }
        };
        // P^T goes to shared memory MN-major: this thread's key kk holds rows
        // [r0, r0 + RH) at bytes [r0, r0 + RH) (E4M3 hi; lo at Rp + r0) or [2 r0, 2 r0 + 2 RH)
        // (bf16) of its row
        auto encode = [&](bool add) {  // add: take the probabilities into l
        const uint32_t pb = base + st * S::kStageBytes;  // over this step's K (read by Q K^T)
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const int kk = kt + 128 * m;  // key within the step
          static_assert(RH == 32 || RH == 16 || RH == 8, "rows per compute warp");
          if (KV == HPA_KV_BF16) {
            uint32_t pw[RH / 2];  // rows (r0 + e, r0 + e + 1) in word e / 2
#pragma unroll
            for (int e = 0; e < RH; e += 2) {
              const float p0 = exp2f(a[m][e]), p1 = exp2f(a[m][e + 1]);
              if (add) upk(add2(pk(lsum[e], lsum[e + 1]), pk(p0, p1)), lsum[e], lsum[e + 1]);
              pw[e / 2] = pack_bf16(p0, p1);
            }
#pragma unroll
            for (int c = 0; c < RH / 8; ++c)
              sts128(pb + mnmaj(kk, 2 * r0 + 16 * c, S::kPSW), pw[4 * c], pw[4 * c + 1],
                     pw[4 * c + 2], pw[4 * c + 3]);
          } else {
            uint32_t hw[RH / 4], lw[RH / 4];  // rows r0 + e4 .. r0 + e4 + 3 in word e4 / 4
#pragma unroll
            for (int e4 = 0; e4 < RH; e4 += 4) {
              uint32_t hi = 0, lo = 0;
#pragma unroll
              for (int e = 0; e < 4; e += 2) {
                const int a0 = e4 + e;
                const float p0 = exp2f(a[m][a0]);
                const float p1 = exp2f(a[m][a0 + 1]);
                if (add) upk(add2(pk(lsum[a0], lsum[a0 + 1]), pk(p0, p1)), lsum[a0], lsum[a0 + 1]);
                // hi = e4m3(p), lo = e4m3(p - hi), the residual taken in f16 (exact there)
                const uint32_t pf = pack_f16(p0, p1);
                const uint16_t h2 = f16x2_to_e4m3x2(pf);
                const uint32_t hh = e4m3x2_to_f16x2(h2);
                const __half2 rr2 = __hsub2(*reinterpret_cast<const __half2 *>(&pf),
                                            *reinterpret_cast<const __half2 *>(&hh));
                const uint16_t l2 = f16x2_to_e4m3x2(*reinterpret_cast<const uint32_t *>(&rr2));
                hi |= static_cast<uint32_t>(h2) << (8 * e);
                lo |= static_cast<uint32_t>(l2) << (8 * e);
              }
              hw[e4 / 4] = hi;
              lw[e4 / 4] = lo;
            }
            if constexpr (RH >= 16) {
#pragma unroll
              for (int c = 0; c < RH / 16; ++c) {
                sts128(pb + mnmaj(kk, r0 + 16 * c, S::kPSW), hw[4 * c], hw[4 * c + 1],
                       hw[4 * c + 2], hw[4 * c + 3]);
                sts128(pb + mnmaj(kk, kRp + r0 + 16 * c, S::kPSW), lw[4 * c], lw[4 * c + 1],
                       lw[4 * c + 2], lw[4 * c + 3]);
              }
            } else {
              sts64(pb + mnmaj(kk, r0, S::kPSW), hw[0], hw[1]);
              sts64(pb + mnmaj(kk, kRp + r0, S::kPSW), lw[0], lw[1]);
            }
          }
        }
        };
        scores();
        // Every read of S[b] is done (a moved reference recovers x from a): Q K^T of a
        // later step may overwrite it while this step votes and encodes.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * (B_S_FREE + b));
        // A reference moves only when some score exceeds it by more than the slack, i.e.
        // when a > kSlack + kPOff, and always while a row has none.
        float amax = a[0][0];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int e = 0; e < RH; ++e) amax = fmaxf(amax, a[m][e]);
        const bool flag = amax > kSlack + kPOff || unref != 0;
        // The 4 warps that share this warp's rows agree through an mbarrier of their own
        // (bounded waits, never named barriers: a warp that gives up must not leave the
        // others waiting without a limit).
        const bool any = __any_sync(kFull, flag);
        if (lane == 0) {
          flags[b * 16 + w] = any;  // w = 4 hf + qd
          mbar_arrive(bars + 8 * (B_FLAG + 4 * b + hf));
        }
        // Wait out the P V of two steps back.  P^T lives in this step's own stage, so no
        // buffer depends on it; the wait keeps this thread's parity waits on PV_DONE[b]
        // in order (each of its uses waited, so a later parity wait cannot mistake an
        // older phase for the one it expects) and bounds how far the compute warps run
        // ahead of P V.
        if (i >= 2 && (*abort_flag ||
                       !mbar_wait_bounded_rolled(bars + 8 * (B_PV_DONE + b), ((i - 2) >> 1) & 1))) {
          ok = false;
          break;
        }
        // While the vote completes, a warp with no score past the slack writes its
        // probabilities against the reference as it stands.  If the vote moves the
        // reference, they are written again; l already holds them, and the rescale by
        // alpha = 2^(bo - bn) turns 2^(x - bo) into 2^(x - bn).
        if (!any) encode(true);
        if (*abort_flag || !mbar_wait_bounded_rolled(bars + 8 * (B_FLAG + 4 * b + hf), (i >> 1) & 1)) {
          ok = false;
          break;
        }
        int moved = 0;
#pragma unroll
        for (int x4 = 0; x4 < 4; ++x4) moved |= flags[b * 16 + 4 * hf + x4];
        if (moved) {
          // the plain scores x = a + bo = a - nb (S[b] is already released)
#pragma unroll
          for (int e4 = 0; e4 < RH; e4 += 4) {
            float nb4[4];
            nbias4(e4, nb4);
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
              for (int e1 = 0; e1 < 4; ++e1) a[m][e4 + e1] -= nb4[e1];
          }
          float *sm = stepmax + (n_moved & 1) * 4 * 64;
#pragma unroll
          for (int e = 0; e < RH; ++e) {
            float v = a[0][e];
#pragma unroll
            for (int m = 1; m < MT; ++m) v = fmaxf(v, a[m][e]);
            const float mx = warp_max(v);
            if (lane == 0) sm[qd * 64 + r0 + e] = mx;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bars + 8 * (B_SMAX + hf));
          if (*abort_flag || !mbar_wait_bounded_rolled(bars + 8 * (B_SMAX + hf), n_moved & 1)) {
            ok = false;
            break;
          }
          ++n_moved;
          float alpha[RH];
          bool rescale = false;
          uint32_t nunref = 0;
#pragma unroll
          for (int e4 = 0; e4 < RH; e4 += 4) {
            float b4[4], bn4[4];
            bias4(e4, b4);
#pragma unroll
            for (int e1 = 0; e1 < 4; ++e1) {
              const int e = e4 + e1, r = r0 + e;
              const float bo = (unref >> e) & 1u ? -CUDART_INF_F : b4[e1];
              // new reference: the max of the row so far (never below the old one)
              const float mn = fmaxf(fmaxf(fmaxf(sm[r], sm[64 + r]), fmaxf(sm[128 + r], sm[192 + r])),
                                     bo + kPOff);
              const float bn = mn - kPOff;
              alpha[e] = bn == bo ? 1.f : exp2f(bo - bn);  // 0 from -inf
              rescale |= alpha[e] != 1.f;
              lsum[e] *= alpha[e];
              const bool none = bn == -CUDART_INF_F;  // a row with no visible key yet
              nunref |= (none && (r < R) ? 1u : 0u) << e;
              bn4[e1] = none ? 0.f : bn;
#pragma unroll
              for (int m = 0; m < MT; ++m) a[m][e] -= bn4[e1];
            }
            if constexpr (S::kBiasInSmem) __syncwarp();  // every lane has read the old values
#pragma unroll
            for (int e1 = 0; e1 < 4; ++e1) bias_set(e4 + e1, bn4[e1]);
          }
          unref = nunref;
          if constexpr (S::kBiasInSmem) __syncwarp();
          if (jp > 0 && __any_sync(kFull, rescale)) {
            // O holds the earlier steps of this segment: wait for the last P V, then
            // rescale this warp's rows of it in TMEM (lane = output dim kt)
            const int pi = i - 1;
            if (*abort_flag ||
                !mbar_wait_bounded_rolled(bars + 8 * (B_PV_DONE + (pi & 1)), (pi >> 1) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int part = 0; part < S::kNS / kRp; ++part)  // O (and its lo half)
#pragma unroll
              for (int c = 0; c < RH / 8; ++c) {
                const uint32_t col = lane_t + S::kOCol + part * kRp + r0 + 8 * c;
                float o[8];
                tc_ld8(col, o);
                tc_wait_ld();
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] *= alpha[8 * c + e];
                tc_st8(col, o);
              }
            tc_wait_st();
          }
          encode(any);  // l takes them now only if this warp did not write them above
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const int kk = kt + 128 * m;  // key within the step
          // V rows of keys past the request (or of a missing page) must be finite: zero them
          if (hf == 0 && (key0 + 128 * m >= pg1 * PAGE || key0 + 128 * m >= L)) {
            uint8_t *vr = smem + st * S::kStageBytes + S::kKStep + (kk >> 3) * 1024 + (kk & 7) * 128;
            const int4 z = make_int4(0, 0, 0, 0);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              reinterpret_cast<int4 *>(vr)[c] = z;
              if (KV == HPA_KV_BF16) reinterpret_cast<int4 *>(vr + S::kPPS * 8192)[c] = z;
            }
          }
        }
        fence_proxy_async_smem();  // generic writes before the MMA reads them
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * (B_P_FULL + b));

        if (jp == nsteps - 1) {
          // ---- segment end: l per row (sum over the 128 key slots), then O / l for
          // this warp's rows, this thread's dim kt
#pragma unroll
          for (int e = 0; e < RH; ++e) {
            float v = lsum[e];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
            if (lane == 0) lred[qd * 64 + r0 + e] = v;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bars + 8 * (B_LRED + hf));
          if (*abort_flag || !mbar_wait_bounded_rolled(bars + 8 * (B_LRED + hf), n_seg & 1) ||
              !mbar_wait_bounded_rolled(bars + 8 * (B_PV_DONE + b), (i >> 1) & 1)) {
            ok = false;
            break;
          }
          ++n_seg;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < RH / 8; ++c) {
            float o[8];
            tc_ld8(lane_t + S::kOCol + r0 + 8 * c, o);
            if (KV == HPA_KV_E4M3) {  // O = O(P hi) + O(P lo)
              float u[8];
              tc_ld8(lane_t + S::kOCol + kRp + r0 + 8 * c, u);
              tc_wait_ld();
#pragma unroll
              for (int e = 0; e < 8; ++e) o[e] += u[e];
            }
            tc_wait_ld();
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int r = r0 + 8 * c + e;
              const float l = lred[r] + lred[64 + r] + lred[128 + r] + lred[192 + r];
              if (r < R) {
                const int j = jrow[r], g = r - j * G;
                const int64_t row = (static_cast<int64_t>(s) * q_len + j) * p.Hq + h * G + g;
                p.partial_o[row * HEAD_DIM + kt] = l > 0.f ? o[e] / l * vsc : 0.f;
                if (kt == 8 * c + e) {  // one thread per row writes its lse
                  float b4[4];
                  bias4((8 * c + e) & ~3, b4);
                  p.partial_lse[row] =
                      l > 0.f ? (b4[(8 * c + e) & 3] + log2f(l)) * 0.69314718055994531f
                              : -CUDART_INF_F;
                }
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(bars + 8 * B_O_FREE);              // O may be overwritten
            mbar_arrive(bars + 8 * (B_Q_EMPTY + slot));    // the query slot may be refilled
          }
        }
        ++i;
      }
    }
    if (!ok && t == 0) {
      status_or(p.tm, HPA_STATUS_TIMEOUT);
      *abort_flag = 1;
    }
  }
};

template <int KV, int NC>
__global__ void __launch_bounds__(TcSmem<KV, NC>::kThreads, 1)
    decode_attn_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                          const __grid_constant__ CUtensorMap tmv, const AttnParams p) {
  using S = TcSmem<KV, NC>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int c = blockIdx.x, h = blockIdx.y;
  __shared__ int hdr[4];  // go, tile, s_begin, s_end
  const uint32_t base = smem_u32(smem), bars = base + S::kBars;
  // optional per-CTA timestamps: entry, map read, last segment stored, smid | segments << 32
  unsigned long long *trace =
      p.trace ? p.trace + 4 * (static_cast<int64_t>(h) * p.C + c) : nullptr;
  if (trace && threadIdx.x == 0) trace[0] = globaltimer_ns();
  pdl_wait();
  if (threadIdx.x == 0) {
    const int32_t *tm = p.tm;
    const int tile = tm[TM_TILE];
    int go = tm[TM_STATUS] == 0;
    if (go && (tm[TM_B] != p.B || tm[TM_C] != p.C || tile <= 0 || tile % PAGE != 0)) {
      if (c == 0 && h == 0) status_or(p.tm, HPA_STATUS_MISMATCH);
      go = 0;
    }
    if (go && !map_ranges_ok(tm, p.lay, p.B, p.C, c)) {
      status_or(p.tm, HPA_STATUS_BAD_MAP);
      go = 0;
    }
    hdr[1] = tile;
    hdr[2] = go ? tm[p.lay.cta_seg + c] : 0;
    hdr[3] = go ? tm[p.lay.cta_seg + c + 1] : 0;
    hdr[0] = go && hdr[2] < hdr[3];
    // q_full q_empty s_full s_free p_full pv_done o_free drain flag smax lred
    constexpr int CW = S::kCW;
    // q_full q_empty s_full s_free p_full pv_done o_free drain; then per row group
    // (4 warps each) flag[2][4] smax[4] lred[4]
    const int counts[30] = {32, 32, 1 + CW, 1 + CW, 1, 1, CW, CW, CW, CW, 1, 1, CW, 2,
                            4, 4, 4, 4, 4, 4, 4, 4, 4, 4, 4, 4, 4, 4, 4, 4};
    for (int i = 0; i < 30; ++i) mbar_init(bars + 8 * i, counts[i]);
    for (int i = 0; i < S::kStages; ++i) {
      mbar_init(bars + 8 * (B_KV_FULL + i), 1);                 // TMA bytes
      mbar_init(bars + 8 * (S::kKvEmpty + i), 1);      // MMA commit
    }
    for (int r = 0; r < 64; ++r) reinterpret_cast<int *>(smem + S::kJRow)[r] = r / p.G;
    *reinterpret_cast<int *>(smem + S::kAbort) = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  if (trace && threadIdx.x == 0) {
    trace[1] = globaltimer_ns();
    trace[3] = smid() | (static_cast<unsigned long long>(hdr[3] - hdr[2]) << 32);
  }
  if (!hdr[0]) {  // bad map, or a partition with no tiles
    if (trace && threadIdx.x == 0) trace[2] = globaltimer_ns();
    return;
  }
  if (threadIdx.x < 32) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     base + S::kTmem),
                 "r"(S::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + S::kTmem);
  const int tile = hdr[1], s_begin = hdr[2], s_end = hdr[3];
  const int warp = threadIdx.x >> 5;
  if (warp < S::kCW)
    Tc<KV, NC>::compute(p, smem, s_begin, s_end, tmem, h);
  else if (warp == S::kCW)
    Tc<KV, NC>::producer(p, &tmk, &tmv, smem, s_begin, s_end, tile, h);
  else if (warp == S::kCW + 1 && (threadIdx.x & 31) == 0)
    Tc<KV, NC>::qk_issuer(p, smem, s_begin, s_end, tile, tmem);
  else if (warp == S::kCW + 2 && (threadIdx.x & 31) == 0)
    Tc<KV, NC>::pv_issuer(p, smem, s_begin, s_end, tile, tmem);
  tc_fence_before();
  __syncthreads();
  if (trace && threadIdx.x == 0) trace[2] = globaltimer_ns();  // every segment stored
  // both issuers have committed to the drain barrier: wait (bounded) for their MMAs
  mbar_wait_bounded_rolled(bars + 8 * B_DRAIN, 0, 1000000000ull);
  if (threadIdx.x < 32) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(S::kTmemCols)
                 : "memory");
  }
}

template <int KV, int NC>
cudaError_t launch_tc(const AttnParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                      cudaStream_t s) {
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(decode_attn_tc_kernel<KV, NC>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, TcSmem<KV, NC>::kAlloc);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.C, p.Hkv, 1);
  cfg.blockDim = dim3(TcSmem<KV, NC>::kThreads);
  cfg.dynamicSmemBytes = TcSmem<KV, NC>::kAlloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_attn_tc_kernel<KV, NC>, tmk, tmv, p);
}

template <int KV>
cudaError_t launch_tc_kv(const AttnParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                         cudaStream_t s) {
  switch ((p.rows + 15) / 16) {
    case 1: return launch_tc<KV, 1>(p, tmk, tmv, s);
    case 2: return launch_tc<KV, 2>(p, tmk, tmv, s);
    case 3: return launch_tc<KV, 3>(p, tmk, tmv, s);
    default: return launch_tc<KV, 4>(p, tmk, tmv, s);
  }
}

template <int KV, int NC>
int occupancy_tc(int *ctas) {
  cudaError_t e = cudaFuncSetAttribute(decode_attn_tc_kernel<KV, NC>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TcSmem<KV, NC>::kAlloc);
  if (e != cudaSuccess) return -1;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, decode_attn_tc_kernel<KV, NC>,
                                                    TcSmem<KV, NC>::kThreads,
                                                    TcSmem<KV, NC>::kAlloc);
  return e == cudaSuccess ? 0 : -1;
}

template <int KV>
int occupancy_tc_kv(int rows, int *ctas) {
  switch ((rows + 15) / 16) {
    case 1: return occupancy_tc<KV, 1>(ctas);
    case 2: return occupancy_tc<KV, 2>(ctas);
    case 3: return occupancy_tc<KV, 3>(ctas);
    default: return occupancy_tc<KV, 4>(ctas);
  }
}

}  // namespace

cudaError_t launch_decode_attn_tc(const AttnParams &p, const CUtensorMap &tmk,
                                  const CUtensorMap &tmv, int kv_dtype, cudaStream_t s) {
  return kv_dtype == HPA_KV_BF16 ? launch_tc_kv<HPA_KV_BF16>(p, tmk, tmv, s)
                                 : launch_tc_kv<HPA_KV_E4M3>(p, tmk, tmv, s);
}

int attn_tc_ctas_per_sm(int kv_dtype, int rows, int *ctas) {
  return kv_dtype == HPA_KV_BF16 ? occupancy_tc_kv<HPA_KV_BF16>(rows, ctas)
                                 : occupancy_tc_kv<HPA_KV_E4M3>(rows, ctas);
}

}  // namespace hpa
