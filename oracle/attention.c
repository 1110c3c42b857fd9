/*
 * ORACLE -- test infrastructure only.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg may load this code; the product path
 * never does.  It shares no source with the CUDA library.
 *
 * Plain fp64 GQA decode attention over a paged KV cache, written from its
 * definition:
 *   for request r, query token j, query head g (KV head h = g / (Hq/Hkv)):
 *     s_k   = sm_scale * <q[r][j][g], k_k>        for visible keys k
 *     out   = sum_k exp(s_k - m) v_k / sum_k exp(s_k - m),  m = max_k s_k
 *     lse   = m + ln sum_k exp(s_k - m)
 * The model shape (64 query heads sharing 8 KV heads, head dim 128) is the
 * one in "Hy3 Preview AI Infra 推理优化精读笔记", §2 "模型与问题背景".
 *
 * One call evaluates a list of items (request, key_lo, key_hi): the item sees
 * keys [key_lo, key_hi) of its request.  The full range gives the unsplit
 * result; a tile range gives one split-KV partial, as in the same page,
 * §3.1 "Attention：动态切分和负载均衡" (方案 steps 4-5), where each CTA
 * produces partial results over its tiles for a later merge.
 *
 * Readings where the pages are silent:
 *  - query token j of q_len new tokens sits at position L - q_len + j and sees
 *    keys [0, L - q_len + 1 + j) (causal, bottom-right aligned);
 *  - a row that sees no key in an item has lse = -inf and out = 0;
 *  - KV elements are bf16, or OCP E4M3 codes times one fp32 scale per KV
 *    head (the pages name "Attention FP8" / C8 without a format).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { KV_BF16 = 0, KV_E4M3 = 1 };

/* bf16 is the upper half of an IEEE binary32. */
static double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP 8-bit E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities;
 * S.1111.111 is NaN; exponent field 0 encodes subnormals m/8 * 2^-6. */
static double e4m3_to_double(uint8_t b) {
    int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexp((double)m / 8.0, -6);
    else mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

double oracle_bf16_to_double(uint16_t b) { return bf16_to_double(b); }
double oracle_e4m3_to_double(uint8_t b) { return e4m3_to_double(b); }

typedef struct {
    const uint16_t *q;
    const uint8_t *k_pool, *v_pool;
    int kv_dtype;
    const float *k_scale, *v_scale;
    const int32_t *seq_lens, *page_indptr, *page_indices;
    int64_t num_pages;
    int page_size, B, q_len, Hq, Hkv, d;
    double sm_scale;
    int n_items;
    const int32_t *items; /* [n_items][3] = {req, key_lo, key_hi} */
    double *out, *lse;    /* [n_items][q_len][Hq][d], [n_items][q_len][Hq] */
    int64_t next;         /* work counter over (item, kv head) */
    pthread_mutex_t mu;
    int error;
} job_t;

/* Read element i of the key/value vector of key `key` of request r, KV head h. */
static void load_kv(const job_t *J, const uint8_t *pool, const float *scale, int r, int h,
                    int key, double *dst) {
    int32_t page = J->page_indices[J->page_indptr[r] + key / J->page_size];
    int64_t off = (((int64_t)page * J->Hkv + h) * J->page_size + key % J->page_size) * J->d;
    for (int i = 0; i < J->d; ++i) {
        if (J->kv_dtype == KV_BF16) {
            uint16_t b;
            memcpy(&b, pool + 2 * (off + i), 2);
            dst[i] = bf16_to_double(b);
        } else {
            dst[i] = e4m3_to_double(pool[off + i]) * (double)scale[h];
        }
    }
}

static void run_unit(job_t *J, int item, int h, double *qv, double *kv, double *scores,
                     double *acc) {
    const int G = J->Hq / J->Hkv, rows = J->q_len * G, d = J->d;
    const int r = J->items[3 * item], klo = J->items[3 * item + 1], khi = J->items[3 * item + 2];
    const int L = J->seq_lens[r], n = khi - klo;

    /* query rows of this KV head: row = j * G + g */
    for (int j = 0; j < J->q_len; ++j)
        for (int g = 0; g < G; ++g)
            for (int i = 0; i < d; ++i)
                qv[(j * G + g) * d + i] =
                    bf16_to_double(J->q[(((int64_t)r * J->q_len + j) * J->Hq + h * G + g) * d + i]);

    /* scores; invisible keys get -inf */
    for (int t = 0; t < n; ++t) {
        int key = klo + t;
        load_kv(J, J->k_pool, J->k_scale, r, h, key, kv);
        for (int row = 0; row < rows; ++row) {
            int j = row / G;
            int limit = L - J->q_len + 1 + j;
            double s = -INFINITY;
            if (key < limit) {
                s = 0.0;
                for (int i = 0; i < d; ++i) s += qv[row * d + i] * kv[i];
                s *= J->sm_scale;
            }
            scores[(int64_t)row * n + t] = s;
        }
    }

    /* softmax with max subtraction, then the weighted sum of values */
    double m[64], l[64];
    for (int row = 0; row < rows; ++row) {
        double mx = -INFINITY, sum = 0.0;
        for (int t = 0; t < n; ++t) mx = fmax(mx, scores[(int64_t)row * n + t]);
        if (mx != -INFINITY)
            for (int t = 0; t < n; ++t) {
                double p = exp(scores[(int64_t)row * n + t] - mx);
                scores[(int64_t)row * n + t] = p;
                sum += p;
            }
        m[row] = mx;
        l[row] = sum;
        for (int i = 0; i < d; ++i) acc[row * d + i] = 0.0;
    }
    for (int t = 0; t < n; ++t) {
        load_kv(J, J->v_pool, J->v_scale, r, h, klo + t, kv);
        for (int row = 0; row < rows; ++row) {
            if (m[row] == -INFINITY) continue;
            double p = scores[(int64_t)row * n + t];
            if (p == 0.0) continue;
            for (int i = 0; i < d; ++i) acc[row * d + i] += p * kv[i];
        }
    }
    for (int row = 0; row < rows; ++row) {
        int j = row / G, g = row % G;
        int64_t o = (((int64_t)item * J->q_len + j) * J->Hq + h * G + g);
        for (int i = 0; i < d; ++i)
            J->out[o * d + i] = (m[row] == -INFINITY) ? 0.0 : acc[row * d + i] / l[row];
        J->lse[o] = (m[row] == -INFINITY) ? -INFINITY : m[row] + log(l[row]);
    }
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    const int G = J->Hq / J->Hkv, rows = J->q_len * G;
    int64_t maxn = 1;
    for (int it = 0; it < J->n_items; ++it) {
        int64_t n = J->items[3 * it + 2] - J->items[3 * it + 1];
        if (n > maxn) maxn = n;
    }
    double *qv = malloc(sizeof(double) * rows * J->d);
    double *kv = malloc(sizeof(double) * J->d);
    double *acc = malloc(sizeof(double) * rows * J->d);
    double *scores = malloc(sizeof(double) * rows * maxn);
    if (!qv || !kv || !acc || !scores) {
        pthread_mutex_lock(&J->mu);
        J->error = -2;
        pthread_mutex_unlock(&J->mu);
    } else {
        for (;;) {
            pthread_mutex_lock(&J->mu);
            int64_t u = J->next++;
            pthread_mutex_unlock(&J->mu);
            if (u >= (int64_t)J->n_items * J->Hkv) break;
            run_unit(J, (int)(u / J->Hkv), (int)(u % J->Hkv), qv, kv, scores, acc);
        }
    }
    free(qv);
    free(kv);
    free(acc);
    free(scores);
    return NULL;
}

/* Returns 0 on success; -1 for an invalid argument (nothing computed); -2 on
 * allocation failure.  n_threads <= 0 uses every online host core. */
int oracle_attention(const uint16_t *q, const void *k_pool, const void *v_pool, int kv_dtype,
                     const float *k_scale, const float *v_scale, const int32_t *seq_lens,
                     const int32_t *page_indptr, const int32_t *page_indices, int64_t num_pages,
                     int page_size, int B, int q_len, int Hq, int Hkv, int d, double sm_scale,
                     int n_items, const int32_t *items, int n_threads, double *out, double *lse) {
    if (!q || !k_pool || !v_pool || !seq_lens || !page_indptr || !page_indices || !items ||
        !out || !lse)
        return -1;
    if (B <= 0 || q_len <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || page_size <= 0)
        return -1;
    if ((Hq / Hkv) * q_len > 64) return -1;
    if (kv_dtype != KV_BF16 && kv_dtype != KV_E4M3) return -1;
    if (kv_dtype == KV_E4M3 && (!k_scale || !v_scale)) return -1;
    for (int it = 0; it < n_items; ++it) {
        int r = items[3 * it], lo = items[3 * it + 1], hi = items[3 * it + 2];
        if (r < 0 || r >= B || lo < 0 || hi < lo || hi > seq_lens[r]) return -1;
    }
    for (int r = 0; r < B; ++r) {
        if (seq_lens[r] < q_len) return -1;
        int64_t need = (seq_lens[r] + page_size - 1) / page_size;
        if (page_indptr[r + 1] - page_indptr[r] < need) return -1;
        for (int64_t p = page_indptr[r]; p < page_indptr[r] + need; ++p)
            if (page_indices[p] < 0 || page_indices[p] >= num_pages) return -1;
    }
    job_t J = {q, k_pool, v_pool, kv_dtype, k_scale, v_scale, seq_lens, page_indptr,
               page_indices, num_pages, page_size, B, q_len, Hq, Hkv, d, sm_scale, n_items,
               items, out, lse, 0};
    pthread_mutex_init(&J.mu, NULL);
    J.error = 0;
    if (n_threads <= 0) n_threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    pthread_t th[256];
    int started = 0;
    for (int i = 0; i < n_threads; ++i)
        if (pthread_create(&th[started], NULL, worker, &J) == 0) ++started;
    if (started == 0) worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    pthread_mutex_destroy(&J.mu);
    return J.error;
}
