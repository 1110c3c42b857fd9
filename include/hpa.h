/*
 * hpa.h -- load-balanced split-KV GQA decode attention for NVIDIA GB300 (sm_103a).
 *
 * C ABI.  Every pointer argument named *_dev is a device pointer allocated by
 * the caller; the library never allocates or frees memory and never
 * synchronises a stream.  All work is enqueued on the caller's stream in
 * stream order, so the three calls below can be captured in a CUDA graph.
 *
 * The method (sources are web pages, cited by title and section):
 *   [Notes §3.1]  "Hy3 Preview AI Infra 推理优化精读笔记", §3.1 "Attention：动态切分和
 *                 负载均衡" -- cut every request's KV into uniform tiles, join all
 *                 tiles into one stream, give each CTA an equal (or +1) budget of
 *                 it, build a task map before the step, have the attention
 *                 kernel take its tiles from the map, merge split results in a
 *                 combine kernel.  Worked example: lengths 1024/5120/2048, tile
 *                 512 -> 2/10/4 tiles, 4 CTAs x 4 tiles, the long request spans
 *                 CTAs.
 *   [HPC-Ops §二.1] "腾讯混元AI Infra进化：HPC-Ops推理核心算子全面升级", §二.1
 *                 "Attention：动态调度负载均衡" -- a Task Assign module builds the
 *                 map once per inference step; the attention kernel of every
 *                 layer reads it; a Combine kernel merges the split-KV results.
 *   [Stack §二.1]  "大模型推理性能优化新范式：Hy3架构下的全栈优化技术拆解", §二.1 --
 *                 budget base = T / C, the first T % C CTAs get one more tile.
 *   [Notes §2]    same notes page, §2 -- 64 query heads, 8 KV heads, head dim 128.
 *
 * Units used below: B requests; L_r the KV length of request r (counting its
 * q_len new tokens); T the total number of tiles; C = num_ctas, the number of
 * partitions of the tile stream; each partition runs once per KV head, so
 * the attention grid has C x Hkv CTAs.
 *
 * Error behaviour: every call validates its host-visible arguments first and
 * returns a negative HPA_ERR_* code without launching anything when one is
 * wrong.  Problems only the device can see (sequence lengths, page ids, a
 * task map built for another shape or corrupted after it was built, a
 * pipeline wait that ran past its time bound) set bits in the task map's
 * status word (int32 word 6 of the map, HPA_STATUS_*); the attention kernel
 * then does no work for what it cannot trust and the combine kernel writes
 * NaN to every output element, so a bad step cannot pass silently.  The
 * kernels check every index they take from the map before following it, so
 * a corrupted map is reported rather than read or written out of bounds.
 * Asynchronous CUDA faults surface at the caller's next sync.
 */
#ifndef HPA_H
#define HPA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the runtime's stream handle); NULL is the legacy default stream. */
typedef struct CUstream_st *hpa_stream_t;

/* ---- return codes (host) ---- */
#define HPA_OK 0
#define HPA_ERR_INVALID (-1)     /* NULL pointer or out-of-range size; nothing launched */
#define HPA_ERR_UNSUPPORTED (-2) /* a shape these kernels do not implement */
#define HPA_ERR_WORKSPACE (-3)   /* task map buffer smaller than required */
#define HPA_ERR_ALIGN (-4)       /* a pointer lacks the alignment stated below */
#define HPA_ERR_CUDA (-5)        /* a CUDA runtime call or launch failed */
#define HPA_ERR_NOALLOC_CAPACITY (-6) /* the problem needs more than the fixed no-alloc scratch */

/* ---- status bits written by the kernels into task map word 6 ---- */
#define HPA_STATUS_BAD_SEQLEN 1 /* some L_r < 1 (plan) or L_r < q_len (attention) */
#define HPA_STATUS_MISMATCH 2   /* map built for another B / num_ctas / tile */
#define HPA_STATUS_BAD_PAGE 4   /* a page id outside [0, num_pages); page 0 was read instead */
#define HPA_STATUS_TIMEOUT 8    /* a shared-memory pipeline wait exceeded ~2 s; CTA gave up */
#define HPA_STATUS_OVERFLOW 16  /* total tile count does not fit int32 */
#define HPA_STATUS_BAD_MAP 32   /* a malformed map: a partition's segment range, a segment row
                                   (request, owner, tile range) or a request's segment range
                                   out of bounds; the row was skipped, never followed */

/* ---- KV element types ---- */
#define HPA_KV_BF16 0 /* bfloat16 */
#define HPA_KV_E4M3 1 /* OCP FP8 E4M3 code; value = code * scale[kv head] */

/*
 * Task map: an opaque int32 blob in device memory, written by hpa_plan or
 * hpa_plan_static and read by hpa_decode_attn and hpa_combine.  One map
 * serves every layer of a decode step ([HPC-Ops §二.1]).  Layout (int32 words):
 *   [0,16)  header: T, base, rem, C, B, S (segments), status, tile, kind
 *           (0 dynamic / 1 static / 2 token-weighted), splits, S_cap, 0...
 *   lens[B]            copy of the sequence lengths
 *   cu_tiles[B+1]      exclusive running sum of tiles per request
 *   cta_begin[C+1]     first stream tile of each partition
 *   cta_seg[C+1]       first segment of each partition
 *   seg_off[B+1]       first segment of each request
 *   (padding to a multiple of 4 words)
 *   seg[S_cap][4]      {request, tile_lo, tile_hi, partition}; tiles are
 *                      request-local, [tile_lo, tile_hi); unused rows are -1.
 * A segment is the part of one request that one partition owns.
 */

/* Bytes of the dynamic task map for B requests over num_ctas partitions
 * (segment capacity B + num_ctas - 1).  0 if an argument is out of range. */
size_t hpa_taskmap_bytes(int32_t B, int32_t num_ctas);

/* Segment capacity of the dynamic map: B + num_ctas - 1 (0 if out of range).
 * partial_o needs capacity * q_len * Hq * d floats, partial_lse capacity *
 * q_len * Hq floats. */
int32_t hpa_max_segments(int32_t B, int32_t num_ctas);

/* Static comparator: num_ctas = B * splits partitions, capacity B * splits. */
int32_t hpa_static_num_ctas(int32_t B, int32_t splits);
size_t hpa_static_taskmap_bytes(int32_t B, int32_t splits);

/* Partitions per KV head that fill the current device once with the kernel
 * hpa_decode_attn picks for this shape: hpa_default_num_ctas_mma up to 16
 * query rows per KV head (G * q_len), hpa_default_num_ctas_tc above.  Returns
 * <= 0 on a CUDA error or unsupported arguments. */
int32_t hpa_default_num_ctas(int32_t Hq, int32_t Hkv, int32_t q_len, int32_t kv_dtype);

/* Partitions per KV head for hpa_decode_attn_mma: SMs x resident CTAs per SM /
 * (Hkv x query-row groups), at least 1, where a group is 16 of the G * q_len
 * query rows of a KV head. */
int32_t hpa_default_num_ctas_mma(int32_t Hq, int32_t Hkv, int32_t q_len, int32_t kv_dtype);

/*
 * hpa_plan -- the Task Assign step ([Notes §3.1] steps 1-4, [HPC-Ops §二.1],
 * [Stack §二.1]).  One device kernel:
 *   n_r = ceil(L_r / tile); cu_tiles = exclusive scan of n_r; T = cu_tiles[B];
 *   base = T / C, rem = T % C; partition c owns stream tiles
 *   [c*base + min(c, rem), (c+1)*base + min(c+1, rem)); its range is split at
 *   request boundaries into segments.
 * seq_lens_dev: int32[B] device, L_r >= 1.  tile: a positive multiple of 64
 * (the page size).  num_ctas >= 1 (more partitions than tiles leaves the
 * surplus empty).  taskmap_dev: >= hpa_taskmap_bytes(B, num_ctas) bytes,
 * 16-byte aligned.
 */
int hpa_plan(const int32_t *seq_lens_dev, int32_t B, int32_t tile, int32_t num_ctas,
             void *taskmap_dev, size_t taskmap_bytes, hpa_stream_t stream);

/*
 * hpa_plan_weighted -- the token-weighted variant of hpa_plan (a reading the
 * pages leave open: a partial last tile costs its fill, not a whole tile).
 * Same stream, same contiguous partitions and map format (kind 2), with
 * budgets in keys: with K = sum L_r, P_t the keys before stream tile t and w_t
 * the keys in it, tile t goes to partition floor(C (2 P_t + w_t) / (2 K)) --
 * the partition whose equal share of the key stream holds the tile's middle
 * key.  Header words base / rem hold K / C and K % C.  Sizes as hpa_plan;
 * requires (B + C) small enough for the plan's 40 KB shared-memory staging
 * (about B + C <= 3400), else HPA_ERR_UNSUPPORTED; K > 2^40 sets
 * HPA_STATUS_OVERFLOW.
 */
int hpa_plan_weighted(const int32_t *seq_lens_dev, int32_t B, int32_t tile, int32_t num_ctas,
                      void *taskmap_dev, size_t taskmap_bytes, hpa_stream_t stream);

/*
 * hpa_plan_static -- the static split-KV comparator the pages contrast the
 * method with ([Notes §3.1] 问题): request r is cut into min(splits, n_r)
 * contiguous chunks of near-equal tile counts (the first n_r % chunks get
 * one more); partition r * splits + s owns chunk s, or nothing.  Same map
 * format, so the same attention and combine kernels run it.
 * taskmap_dev: >= hpa_static_taskmap_bytes(B, splits) bytes.
 */
int hpa_plan_static(const int32_t *seq_lens_dev, int32_t B, int32_t tile, int32_t splits,
                    void *taskmap_dev, size_t taskmap_bytes, hpa_stream_t stream);

/*
 * hpa_decode_attn -- the split-KV attention kernel ([Notes §3.1] steps 4-5).
 * Up to 16 query rows per KV head (G * q_len <= 16: one new token at any
 * GQA ratio up to 16, or two at 8 heads per KV head) it runs the kernel
 * described here, which is the one that streams the KV at the copy peak
 * there; above 16 rows (MTP with several draft tokens) it runs the same step
 * as hpa_decode_attn_tc, which takes all rows in one pass.  Size num_ctas with
 * hpa_default_num_ctas, which follows the same choice.  hpa_decode_attn_mma
 * runs the kernel described here at any row count.
 *
 * Grid num_ctas x Hkv x ceil(G q_len / 16); the CTA of (partition c, KV
 * head h, row group z) walks c's segments in order and, for each, computes
 * over the segment's keys
 *   s = sm_scale * q . k,  m = max s,  l = sum exp(s - m),  o = sum exp(s - m) v / l
 * for query rows [16 z, 16 z + 16) of the G * q_len rows (row j * G + g:
 * query head g of the G = Hq / Hkv heads of h, token j of the q_len new ones,
 * which sees keys [0, L_r - q_len + 1 + j)), and writes
 *   partial_o[seg][j][head][d] = o,  partial_lse[seg][j][head] = m + ln l
 * (natural log; -inf and o = 0 for a row that sees no key of the segment).
 *
 * q_dev:        bf16 [B][q_len][Hq][d], 16-byte aligned.
 * k_pool_dev, v_pool_dev: [num_pages][Hkv][page_size][d] of bf16 or E4M3
 *               bytes, 16-byte aligned (read with TMA tensor copies).
 * k_scale_dev, v_scale_dev: fp32 [Hkv] for HPA_KV_E4M3, ignored for bf16.
 *               With E4M3 pages the products run in f16: each query row is
 *               scaled by a power of two that puts its largest |element| in
 *               [2^14, 2^15) (taken back out of the scores), so any finite bf16
 *               query converts exactly, down to 2^-28 of its row's largest.
 * page_indptr_dev: int32 [B+1]; page_indices_dev: int32; key i of request r
 *               is slot i % page_size of page page_indices[page_indptr[r] + i / page_size].
 * Supported: d == 128, page_size == 64, Hq % Hkv == 0, (Hq / Hkv) * q_len <= 64,
 *               num_pages * Hkv < 2^31.  Row groups past the first re-read the
 *               pages (through L2 when they run together).
 * taskmap_dev:  a map from hpa_plan / hpa_plan_static for these B and num_ctas.
 * partial_o_dev: fp32, >= (B + num_ctas - 1) * q_len * Hq * d, 16-byte aligned (one
 *               row per segment; no map has more than B + num_ctas - 1 segments);
 * partial_lse_dev: fp32, >= (B + num_ctas - 1) * q_len * Hq.
 */
int hpa_decode_attn(const void *q_dev, const void *k_pool_dev, const void *v_pool_dev,
                    int32_t kv_dtype, const float *k_scale_dev, const float *v_scale_dev,
                    int64_t num_pages, const int32_t *page_indptr_dev,
                    const int32_t *page_indices_dev, int32_t page_size, int32_t B,
                    int32_t q_len, int32_t Hq, int32_t Hkv, int32_t d, float sm_scale,
                    void *taskmap_dev, int32_t num_ctas, float *partial_o_dev,
                    float *partial_lse_dev, hpa_stream_t stream);
int hpa_decode_attn_mma(const void *q_dev, const void *k_pool_dev, const void *v_pool_dev,
                        int32_t kv_dtype, const float *k_scale_dev, const float *v_scale_dev,
                        int64_t num_pages, const int32_t *page_indptr_dev,
                        const int32_t *page_indices_dev, int32_t page_size, int32_t B,
                        int32_t q_len, int32_t Hq, int32_t Hkv, int32_t d, float sm_scale,
                        void *taskmap_dev, int32_t num_ctas, float *partial_o_dev,
                        float *partial_lse_dev, hpa_stream_t stream);

/*
 * hpa_decode_attn_tc -- the same split-KV attention step ([Notes §3.1] steps
 * 4-5), computed by a kernel that runs both products on the 5th-generation
 * tensor cores (tcgen05.mma with accumulators in tensor memory).  Grid
 * num_ctas x Hkv: one CTA covers all G * q_len query rows of its KV head
 * (up to 64) in a single pass over the keys, where hpa_decode_attn makes one
 * pass per group of 16 rows.  It pays for MTP with more than 16 rows per KV
 * head, and hpa_decode_attn runs it there (on the E4M3 MTP workload at 64/8
 * heads: 1.9x the mma.sync kernel at q_len 3-4, 2.7x at q_len 6, 2.6x at
 * q_len 8).  With up to 16 rows, or with many short segments per partition
 * (hundreds of short requests), the mma.sync kernel is as fast or faster.
 * Arguments, layouts, supported shapes, outputs and errors are exactly those
 * of hpa_decode_attn; the partials feed hpa_combine unchanged.  E4M3 pages
 * enter the MMA as 8-bit operands; the query rows and the probabilities are
 * each carried as two E4M3 terms (about 8 significant bits, as bf16).  Each
 * query row is scaled by a power of two (its largest element into [128, 256))
 * and its residual term by a fixed 16, so rows of any bf16 magnitude are
 * carried exactly as long as their elements lie within about 2^-12 of the
 * row's largest; smaller elements lose bits and those below about 2^-21 of it
 * are dropped (hpa_decode_attn_mma keeps bf16 precision down to 2^-28).
 */
int hpa_decode_attn_tc(const void *q_dev, const void *k_pool_dev, const void *v_pool_dev,
                       int32_t kv_dtype, const float *k_scale_dev, const float *v_scale_dev,
                       int64_t num_pages, const int32_t *page_indptr_dev,
                       const int32_t *page_indices_dev, int32_t page_size, int32_t B,
                       int32_t q_len, int32_t Hq, int32_t Hkv, int32_t d, float sm_scale,
                       void *taskmap_dev, int32_t num_ctas, float *partial_o_dev,
                       float *partial_lse_dev, hpa_stream_t stream);

/* Partitions per KV head that fill the current device once with
 * hpa_decode_attn_tc CTAs (SMs x resident CTAs per SM / Hkv), or -1. */
int32_t hpa_default_num_ctas_tc(int32_t Hq, int32_t Hkv, int32_t q_len, int32_t kv_dtype);

/*
 * hpa_decode_attn_traced -- hpa_decode_attn (the same kernel choice) that
 * also records, for every CTA, four uint64 words at trace_dev[4 * (h * num_ctas
 * + c)]: the %globaltimer (ns) at kernel entry, after the task map was read,
 * after the CTA's last segment was stored, and (smid | segments << 32).  Used
 * to measure SM busy time and the tail idle of the last CTA (the pages watch
 * "attention kernel tail idle", "Hy3 Preview AI Infra 推理优化精读笔记", §3.1
 * 对我们的启发).  trace_dev: device, 8-byte aligned, >= 4 * num_ctas * Hkv *
 * row groups words; CTA (c, h, z) of the mma.sync kernel (up to 16 rows) at
 * word 4 * ((z * Hkv + h) * num_ctas + c), CTA (c, h) of the tcgen05 kernel
 * (above 16 rows, no row-group axis) at word 4 * (h * num_ctas + c).
 */
int hpa_decode_attn_traced(const void *q_dev, const void *k_pool_dev, const void *v_pool_dev,
                           int32_t kv_dtype, const float *k_scale_dev, const float *v_scale_dev,
                           int64_t num_pages, const int32_t *page_indptr_dev,
                           const int32_t *page_indices_dev, int32_t page_size, int32_t B,
                           int32_t q_len, int32_t Hq, int32_t Hkv, int32_t d, float sm_scale,
                           void *taskmap_dev, int32_t num_ctas, float *partial_o_dev,
                           float *partial_lse_dev, uint64_t *trace_dev, hpa_stream_t stream);

/*
 * hpa_decode_attn_allheads -- hpa_decode_attn with the KV heads inside the CTA
 * instead of on a grid axis (the pages do not say how heads map to CTAs,
 * "Hy3 Preview AI Infra 推理优化精读笔记" §3.1 方案 step 3; this is the other
 * reading, kept as an A/B).  Grid num_ctas x 1 x row groups: the CTA of
 * partition c walks c's segments and, for each, every KV head in turn
 * (heads innermost), so num_ctas counts partitions of the tile stream for the
 * whole grid (hpa_default_num_ctas_allheads: SMs x resident CTAs per SM /
 * row groups) and the task map must be planned with that count.  Arguments,
 * layouts, partials and errors are those of hpa_decode_attn; trace_dev is
 * NULL or, as for hpa_decode_attn_traced, 4 uint64 words per CTA at
 * trace_dev[4 * (z * num_ctas + c)].
 */
int hpa_decode_attn_allheads(const void *q_dev, const void *k_pool_dev, const void *v_pool_dev,
                             int32_t kv_dtype, const float *k_scale_dev,
                             const float *v_scale_dev, int64_t num_pages,
                             const int32_t *page_indptr_dev, const int32_t *page_indices_dev,
                             int32_t page_size, int32_t B, int32_t q_len, int32_t Hq,
                             int32_t Hkv, int32_t d, float sm_scale, void *taskmap_dev,
                             int32_t num_ctas, float *partial_o_dev, float *partial_lse_dev,
                             uint64_t *trace_dev, hpa_stream_t stream);
int32_t hpa_default_num_ctas_allheads(int32_t Hq, int32_t Hkv, int32_t q_len, int32_t kv_dtype);

/*
 * hpa_decode_attn_fused -- hpa_decode_attn with the combine folded in (one
 * launch instead of two).  Same arguments and layouts, plus the combine's
 * outputs out_dev (bf16 [B][q_len][Hq][d], 8-byte aligned) and out_lse_dev
 * (fp32 [B][q_len][Hq] or NULL), and arrivals_dev: int32 [B][Hkv][row groups]
 * (hpa_arrivals_elems), zero before the first call.
 *   - A request with one segment is written straight to out_dev.
 *   - Otherwise every CTA stores its partial, then counts itself in
 *     arrivals[r][h][z] with an atomic add (after a fence); the CTA whose add
 *     completes the count merges the request's partials for that KV head,
 *     exactly as hpa_combine does, and resets the counter to zero.  No CTA
 *     waits for another.
 * After a call whose map reports a non-zero status, re-zero arrivals_dev
 * before the next call.  A bad map makes every output NaN, as with
 * hpa_combine.  This is the fused combine the pages' three-module design
 * leaves as a later step ("Hy3 Preview AI Infra 推理优化精读笔记", §3.1 step 5:
 * a combine merges the split-KV results).
 */
size_t hpa_arrivals_elems(int32_t B, int32_t Hq, int32_t Hkv, int32_t q_len);
int hpa_decode_attn_fused(const void *q_dev, const void *k_pool_dev, const void *v_pool_dev,
                          int32_t kv_dtype, const float *k_scale_dev, const float *v_scale_dev,
                          int64_t num_pages, const int32_t *page_indptr_dev,
                          const int32_t *page_indices_dev, int32_t page_size, int32_t B,
                          int32_t q_len, int32_t Hq, int32_t Hkv, int32_t d, float sm_scale,
                          void *taskmap_dev, int32_t num_ctas, float *partial_o_dev,
                          float *partial_lse_dev, void *out_dev, float *out_lse_dev,
                          int32_t *arrivals_dev, hpa_stream_t stream);

/*
 * hpa_combine -- the Combine kernel ([Notes §3.1] step 5, [HPC-Ops §二.1]).
 * For every (request r, token j, head g) over r's segments s:
 *   M = max_s lse_s,  w_s = exp(lse_s - M),
 *   out = sum_s w_s o_s / sum_s w_s  (rounded to bf16),  out_lse = M + ln sum_s w_s.
 * out_dev: bf16 [B][q_len][Hq][d], 8-byte aligned; out_lse_dev: fp32
 * [B][q_len][Hq] or NULL.  d == 128.
 */
int hpa_combine(const float *partial_o_dev, const float *partial_lse_dev, void *taskmap_dev,
                int32_t B, int32_t num_ctas, int32_t q_len, int32_t Hq, int32_t d,
                void *out_dev, float *out_lse_dev, hpa_stream_t stream);

/*
 * hpa_store_kv -- the fused KV-cache writer that feeds the decode path
 * ("Hy3 Preview AI Infra 推理优化精读笔记", §4.1 "Rope + Norm + Hadamard + Quant +
 * Store KV": the element-wise chain after the QKV projection in one pass,
 * written straight to the low-bit cache).  For request r, new token j (at
 * position pos = L_r - q_len + j) and KV head h:
 *   key:   rotate-half RoPE with cos_sin[pos] (cos in columns [0, d/2), sin in
 *          [d/2, d)), then RMSNorm over d (x / sqrt(mean x^2 + eps) * norm_w),
 *          then, if use_hadamard, the orthonormal Sylvester Walsh-Hadamard
 *          transform of order d; stored as bf16, or as E4M3 codes of
 *          x / k_scale[h] (round to nearest even, saturating at +-448);
 *   value: stored as bf16, or as E4M3 codes of v / v_scale[h];
 * into slot pos % page_size of page page_indices[page_indptr[r] + pos / page_size]
 * of k_pool_dev / v_pool_dev ([num_pages][Hkv][page_size][d]).
 * k_new_dev, v_new_dev: bf16 [B][q_len][Hkv][d], 16-byte aligned (pools too).  seq_lens_dev:
 * int32 [B], lengths including the new tokens.  cos_sin_dev: fp32 [max_pos][d],
 * 16-byte aligned.  norm_w_dev: fp32 [d], 16-byte aligned.  d == 128,
 * page_size == 64.  status_dev: optional int32; a position outside
 * [0, max_pos) sets HPA_STATUS_BAD_SEQLEN, a missing or out-of-range page
 * HPA_STATUS_BAD_PAGE, and that token is not written.
 */
int hpa_store_kv(const void *k_new_dev, const void *v_new_dev, const int32_t *seq_lens_dev,
                 const int32_t *page_indptr_dev, const int32_t *page_indices_dev,
                 int64_t num_pages, int32_t page_size, const float *cos_sin_dev, int32_t max_pos,
                 const float *norm_w_dev, float eps, int32_t use_hadamard, int32_t kv_dtype,
                 const float *k_scale_dev, const float *v_scale_dev, void *k_pool_dev,
                 void *v_pool_dev, int32_t B, int32_t q_len, int32_t Hkv, int32_t d,
                 int32_t *status_dev, hpa_stream_t stream);

/*
 * hpa_selftest_wait_timeout -- diagnostic for the failure path of the
 * attention pipeline (no counterpart on the pages).  One thread waits on an
 * mbarrier phase that nothing completes, using the same time-bounded wait
 * as hpa_decode_attn, for limit_ns nanoseconds (1e3 .. 5e9); on expiry it ORs
 * HPA_STATUS_TIMEOUT into status_dev[0] and returns, leaving the context
 * usable.  status_dev: one int32 in device memory, 4-byte aligned.
 */
int hpa_selftest_wait_timeout(int32_t *status_dev, int64_t limit_ns, hpa_stream_t stream);

/*
 * hpa_decode_attn_combine_noalloc -- hpa_decode_attn followed by hpa_combine,
 * for callers that cannot allocate device memory; the pages have no
 * counterpart to it.  Such callers include a plugin running inside another
 * runtime that owns the whole device memory pool and hands out no
 * workspace, and a serving loop that must not call cudaMalloc/cudaFree in the
 * middle of a step (cudaFree synchronises the device; either can fail under
 * memory pressure).  Instead of caller-provided partial_o / partial_lse, the
 * split partials live in one fixed array inside the library's device image,
 * HPA_NOALLOC_SCRATCH_BYTES (16 MiB) per GPU, held by every GPU that loads
 * the library until the process exits.  The call itself allocates nothing.
 *
 * Arguments are those of hpa_decode_attn (minus the partial buffers) and of
 * hpa_combine (out_dev, out_lse_dev), with the same layouts and checks.  The
 * partials need (B + num_ctas - 1) * q_len * Hq * (d + 1) floats; a problem
 * larger than the array returns HPA_ERR_NOALLOC_CAPACITY before any launch
 * (e.g. 64 requests x 2 tokens x 64 heads with 38 partitions uses 6.7 MB).
 *
 * The first call on a device resolves the array's device address with that
 * device current (cudaGetSymbolAddress, which may load the module); make that
 * first call before any stream capture.  The address belongs to the CUDA
 * context that was current, so it is cached per context (keyed by the
 * context's process-unique id): a call under another context of the same
 * device, or after cudaDeviceReset, repeats that set-up once for the new
 * context and should likewise come before any capture there.  All calls
 * share the one array and it keeps the last call's contents: nothing in it
 * needs to start at zero (each call writes every partial it reads), but
 * calls that overlap on the GPU -- on different streams, or from several
 * host threads -- race on it and must be serialised by the caller.
 */
#define HPA_NOALLOC_SCRATCH_BYTES (16u << 20)
int hpa_decode_attn_combine_noalloc(const void *q_dev, const void *k_pool_dev,
                                    const void *v_pool_dev, int32_t kv_dtype,
                                    const float *k_scale_dev, const float *v_scale_dev,
                                    int64_t num_pages, const int32_t *page_indptr_dev,
                                    const int32_t *page_indices_dev, int32_t page_size,
                                    int32_t B, int32_t q_len, int32_t Hq, int32_t Hkv,
                                    int32_t d, float sm_scale, void *taskmap_dev,
                                    int32_t num_ctas, void *out_dev, float *out_lse_dev,
                                    hpa_stream_t stream);

/* Static description of a return code. */
const char *hpa_error_string(int code);

/* The last CUDA error the library saw on this thread (cudaError_t value), 0 if none. */
int hpa_last_cuda_error(void);

#ifdef __cplusplus
}
#endif
#endif /* HPA_H */
