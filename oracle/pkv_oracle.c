/*
 * pkv_oracle.c -- plain fp64 CPU oracle for attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the bench's
 * CPU-baseline / reference arm load this file; the CUDA library never does, and
 * this file includes nothing from it.
 *
 * Every result is the textbook definition written out with plain loops in
 * double precision: no tiling, no online softmax, no reordering.
 *
 *   Scaled dot-product attention, softmax(q K^T * scale) V:
 *     limoncc.com "大语言模型研究15——注意力机制优化之KV缓存" §3.1 (Attention formula);
 *     plumephp.com "KV Cache 优化与注意力机制加速" §1.1.
 *   GQA: query head i reads KV head j = floor(i / m), m = Hq / Hkv consecutive
 *     query heads per group:  limoncc.com §3.3 (equation for j);
 *     same page §4.1 (repeat_kv expands KV head j to heads j*m .. j*m+m-1).
 *   Paged addressing: logical token t of a sequence lives in physical block
 *     block_table[t / bs] at offset t % bs:  plumephp.com §4.3 (BlockTable.get_kv).
 *   Log-sum-exp statistic L = m + log(l):  plumephp.com §2.3 (last lines of the
 *     flash_attention pseudocode).
 *   Causal prefill: query t sees keys 0..t of its own sequence, sequences
 *     delimited by cu_seqlens:  0539edu.com "从KV cache共享到批量调度…" §3.3;
 *     zwjcode.cn "KV Cache 的增量解码" §05 (causal prefill), §13 (mask alignment).
 *
 * Cache layout (chosen by this library, the pages leave it open -- 0539edu.com
 * §2.2): k_cache, v_cache are [NB][Hkv][bs][d] row-major.  Element type is fp32
 * (dtype 0), bf16 given as its raw 16-bit pattern (dtype 1), or fp64 (dtype 2, for
 * the exact values of a dequantised FP8 cache).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2 };

/* bf16 is the upper half of an IEEE binary32: widen by appending 16 zero bits.  fp64
 * caches hold values that no narrower type holds exactly (a dequantised code times its
 * fp32 scale). */
static double elem(const void *base, int dtype, size_t i) {
    if (dtype == ORC_F32) return (double)((const float *)base)[i];
    if (dtype == ORC_F64) return ((const double *)base)[i];
    uint32_t u = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * One query row against n contiguous key/value rows (each d doubles).
 *   s_t = scale * sum_e q_e K[t][e]
 *   M   = max_t s_t
 *   w_t = exp(s_t - M),  W = sum_t w_t
 *   o   = sum_t w_t V[t] / W
 *   lse = M + log W
 * n == 0: o = 0, lse = -inf (no key to attend to).
 * s is caller scratch of n doubles.
 */
static double attend(const double *q, const double *K, const double *V, long n, int d,
                     double scale, double *o, double *s) {
    for (int e = 0; e < d; ++e) o[e] = 0.0;
    if (n <= 0) return -INFINITY;
    double M = -INFINITY;
    for (long t = 0; t < n; ++t) {
        double acc = 0.0;
        for (int e = 0; e < d; ++e) acc += q[e] * K[(size_t)t * d + e];
        s[t] = scale * acc;
        if (s[t] > M) M = s[t];
    }
    double W = 0.0;
    for (long t = 0; t < n; ++t) {
        double w = exp(s[t] - M);
        W += w;
        for (int e = 0; e < d; ++e) o[e] += w * V[(size_t)t * d + e];
    }
    for (int e = 0; e < d; ++e) o[e] /= W;
    return M + log(W);
}

/* ------------------------------------------------------------------ threads */

typedef void (*item_fn)(void *ctx, long item);
typedef struct { item_fn fn; void *ctx; long n_items; int tid, nthreads; } worker_arg;

static void *worker(void *p) {
    worker_arg *a = (worker_arg *)p;
    for (long it = a->tid; it < a->n_items; it += a->nthreads) a->fn(a->ctx, it);
    return NULL;
}

/* Run fn(ctx, item) for item in [0, n_items), statically strided over threads. */
static void run_items(item_fn fn, void *ctx, long n_items, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads == 1 || n_items <= 1) {
        for (long it = 0; it < n_items; ++it) fn(ctx, it);
        return;
    }
    pthread_t th[256];
    worker_arg args[256];
    for (int t = 0; t < nthreads; ++t) {
        args[t] = (worker_arg){fn, ctx, n_items, t, nthreads};
        pthread_create(&th[t], NULL, worker, &args[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------ paged decode */

typedef struct {
    double *out, *lse;
    const float *q;
    const void *kc, *vc;
    int dtype;
    const int32_t *table, *lens;
    int B, Hq, Hkv, d, bs, MBS;
    long NB;
    double scale;
    long chunk;          /* tokens per split-K chunk; <= 0: one pass */
    volatile int bad;    /* set when a table entry or length is out of range */
} decode_ctx;

/* Gather sequence b, KV head j into contiguous K[len][d], V[len][d]. */
static int gather(const decode_ctx *c, int b, int j, long len, double *K, double *V) {
    for (long t = 0; t < len; ++t) {
        long page = t / c->bs, off = t % c->bs;
        long phys = c->table[(size_t)b * c->MBS + page];
        if (phys < 0 || phys >= c->NB) return -1;
        size_t row = (((size_t)phys * c->Hkv + j) * c->bs + off) * c->d;
        for (int e = 0; e < c->d; ++e) {
            K[(size_t)t * c->d + e] = elem(c->kc, c->dtype, row + e);
            V[(size_t)t * c->d + e] = elem(c->vc, c->dtype, row + e);
        }
    }
    return 0;
}

/*
 * Split-K: the tokens [c*C, min((c+1)*C, len)) of each chunk c give a partial
 * (o_c, lse_c) by `attend`; the partials combine as
 *   lse = log sum_c exp(lse_c),   o = sum_c exp(lse_c - lse) o_c.
 * This is the online-softmax rescaling (plumephp.com §2.2, online_softmax_update)
 * applied to whole chunks.  An empty chunk has lse_c = -inf and weight 0.
 */
static double attend_split(const double *q, const double *K, const double *V, long n, int d,
                           double scale, long C, double *o, double *s) {
    long nchunks = (n + C - 1) / C;
    double *lses = (double *)malloc(sizeof(double) * (size_t)(nchunks > 0 ? nchunks : 1));
    double *os = (double *)malloc(sizeof(double) * (size_t)(nchunks > 0 ? nchunks : 1) * d);
    double M = -INFINITY;
    for (long c = 0; c < nchunks; ++c) {
        long t0 = c * C, t1 = t0 + C < n ? t0 + C : n;
        lses[c] = attend(q, K + (size_t)t0 * d, V + (size_t)t0 * d, t1 - t0, d, scale,
                         os + (size_t)c * d, s);
        if (lses[c] > M) M = lses[c];
    }
    for (int e = 0; e < d; ++e) o[e] = 0.0;
    double lse = -INFINITY;
    if (M > -INFINITY) {
        double W = 0.0;
        for (long c = 0; c < nchunks; ++c) W += exp(lses[c] - M);
        lse = M + log(W);
        for (long c = 0; c < nchunks; ++c) {
            double w = exp(lses[c] - lse);
            for (int e = 0; e < d; ++e) o[e] += w * os[(size_t)c * d + e];
        }
    }
    free(lses);
    free(os);
    return lse;
}

static void decode_item(void *p, long item) {
    decode_ctx *c = (decode_ctx *)p;
    int b = (int)(item / c->Hkv), j = (int)(item % c->Hkv);
    long len = c->lens[b];
    int m = c->Hq / c->Hkv;
    if (len < 0 || len > (long)c->MBS * c->bs) { c->bad = 1; return; }
    double *K = (double *)malloc(sizeof(double) * (size_t)(len > 0 ? len : 1) * c->d);
    double *V = (double *)malloc(sizeof(double) * (size_t)(len > 0 ? len : 1) * c->d);
    double *s = (double *)malloc(sizeof(double) * (size_t)(len > 0 ? len : 1));
    double *q = (double *)malloc(sizeof(double) * (size_t)c->d);
    if (gather(c, b, j, len, K, V) != 0) c->bad = 1;
    else {
        for (int i = j * m; i < (j + 1) * m; ++i) {   /* the heads with floor(i/m) == j */
            for (int e = 0; e < c->d; ++e) q[e] = (double)c->q[((size_t)b * c->Hq + i) * c->d + e];
            double *o = c->out + ((size_t)b * c->Hq + i) * c->d;
            double l = c->chunk > 0 ? attend_split(q, K, V, len, c->d, c->scale, c->chunk, o, s)
                                    : attend(q, K, V, len, c->d, c->scale, o, s);
            if (c->lse) c->lse[(size_t)b * c->Hq + i] = l;
        }
    }
    free(K); free(V); free(s); free(q);
}

/*
 * out [B][Hq][d] and lse [B][Hq] (may be NULL) in double; q [B][Hq][d] fp32;
 * block_table int32 [B][MBS]; context_lens int32 [B] (tokens in the cache,
 * including any just appended).  chunk_tokens <= 0: one pass; otherwise split-K
 * with that chunk size.  Returns 0, or -1 if a length or a referenced table
 * entry is out of range (outputs then undefined).
 */
int oracle_paged_decode(double *out, double *lse, const float *q, const void *k_cache,
                        const void *v_cache, int dtype, const int32_t *block_table,
                        const int32_t *context_lens, int B, int Hq, int Hkv, int d, int bs,
                        int MBS, long NB, double scale, long chunk_tokens, int nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || bs <= 0 || MBS < 0) return -1;
    decode_ctx c = {out, lse, q, k_cache, v_cache, dtype, block_table, context_lens,
                    B, Hq, Hkv, d, bs, MBS, NB, scale, chunk_tokens, 0};
    run_items(decode_item, &c, (long)B * Hkv, nthreads);
    return c.bad ? -1 : 0;
}

/* ------------------------------------- queries at the end of the cache */

/*
 * Several queries per sequence over the paged cache, with an optional sliding
 * window.  Sequence b holds L = context_lens[b] tokens in the cache, the
 * queries' own K/V among them, and owns query rows cu_q[b] .. cu_q[b+1]-1.  Its
 * i-th query (nq = cu_q[b+1] - cu_q[b] of them) is the token at position
 * p = L - nq + i and attends the keys lo .. p, causally aligned to the end of
 * the cache (zwjcode.cn "KV Cache 的增量解码" §13: a query sees itself and the
 * keys before it, not the later new tokens).  lo = 0 without a window; with
 * window W > 0 it is max(0, p - W + 1): the most recent W positions
 * (zwjcode.cn §10 "滑动窗口", §15; plumephp.com "KV Cache 优化与注意力机制加速"
 * §5.2).  One query per sequence and no window is the decode of
 * oracle_paged_decode; many queries is a prefill on top of cached context.
 */
typedef struct {
    double *out, *lse;
    const float *q;
    const void *kc, *vc;
    int dtype;
    const int32_t *table, *lens, *cu_q;
    int B, Hq, Hkv, d, bs, MBS;
    long NB;
    double scale;
    long window;
    volatile int bad;
} multi_ctx;

/* Gather tokens [t0, t1) of sequence b, KV head j into K[t1-t0][d], V[t1-t0][d]. */
static int gather_range(const multi_ctx *c, int b, int j, long t0, long t1, double *K, double *V) {
    for (long t = t0; t < t1; ++t) {
        long page = t / c->bs, off = t % c->bs;
        long phys = c->table[(size_t)b * c->MBS + page];
        if (phys < 0 || phys >= c->NB) return -1;
        size_t row = (((size_t)phys * c->Hkv + j) * c->bs + off) * c->d;
        for (int e = 0; e < c->d; ++e) {
            K[(size_t)(t - t0) * c->d + e] = elem(c->kc, c->dtype, row + e);
            V[(size_t)(t - t0) * c->d + e] = elem(c->vc, c->dtype, row + e);
        }
    }
    return 0;
}

static void multi_item(void *p, long item) {
    multi_ctx *c = (multi_ctx *)p;
    int b = (int)(item / c->Hkv), j = (int)(item % c->Hkv);
    long L = c->lens[b], r0 = c->cu_q[b], nq = (long)c->cu_q[b + 1] - c->cu_q[b];
    int m = c->Hq / c->Hkv, d = c->d;
    if (L < 0 || L > (long)c->MBS * c->bs || nq < 0 || nq > L) { c->bad = 1; return; }
    if (nq == 0) return;
    long first = L - nq;   /* position of the first query */
    long lo0 = c->window > 0 ? first - c->window + 1 : 0;
    if (lo0 < 0) lo0 = 0;
    long n = L - lo0;      /* every key any of the queries sees */
    double *K = (double *)malloc(sizeof(double) * (size_t)n * d);
    double *V = (double *)malloc(sizeof(double) * (size_t)n * d);
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double *q = (double *)malloc(sizeof(double) * (size_t)d);
    if (gather_range(c, b, j, lo0, L, K, V) != 0) c->bad = 1;
    else {
        for (long i = 0; i < nq; ++i) {
            long pos = first + i;
            long lo = c->window > 0 ? pos - c->window + 1 : 0;
            if (lo < 0) lo = 0;
            for (int h = j * m; h < (j + 1) * m; ++h) {   /* the heads with floor(h/m) == j */
                size_t row = (size_t)(r0 + i) * c->Hq + h;
                for (int e = 0; e < d; ++e) q[e] = (double)c->q[row * d + e];
                double l = attend(q, K + (size_t)(lo - lo0) * d, V + (size_t)(lo - lo0) * d,
                                  pos - lo + 1, d, c->scale, c->out + row * d, s);
                if (c->lse) c->lse[row] = l;
            }
        }
    }
    free(K); free(V); free(s); free(q);
}

/*
 * out [Tq][Hq][d], lse [Tq][Hq] (may be NULL) in double; q [Tq][Hq][d] fp32;
 * cu_q int32 [B+1] (cu_q[0] = 0, cu_q[B] = Tq); window <= 0: no window.  Table
 * entries of pages no query sees are never read.  Returns 0, or -1 for a bad
 * length, a query count above its length, or a bad table entry that is read.
 */
int oracle_paged_attention(double *out, double *lse, const float *q, const void *k_cache,
                           const void *v_cache, int dtype, const int32_t *block_table,
                           const int32_t *context_lens, const int32_t *cu_q, int B, int Hq, int Hkv,
                           int d, int bs, int MBS, long NB, double scale, long window, int nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || bs <= 0 || MBS < 0) return -1;
    multi_ctx c = {out, lse, q, k_cache, v_cache, dtype, block_table, context_lens, cu_q,
                   B, Hq, Hkv, d, bs, MBS, NB, scale, window, 0};
    run_items(multi_item, &c, (long)B * Hkv, nthreads);
    return c.bad ? -1 : 0;
}

/* ------------------------------------------------- contiguous (no paging) */

/*
 * q [Hq][d], K/V [Hkv][n][d] all double; out [Hq][d], lse [Hq].
 * The same definition without a block table.
 */
void oracle_attend_contiguous(double *out, double *lse, const double *q, const double *K,
                              const double *V, long n, int Hq, int Hkv, int d, double scale) {
    int m = Hq / Hkv;
    double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    for (int i = 0; i < Hq; ++i) {
        int j = i / m;
        double l = attend(q + (size_t)i * d, K + (size_t)j * n * d, V + (size_t)j * n * d, n, d,
                          scale, out + (size_t)i * d, s);
        if (lse) lse[i] = l;
    }
    free(s);
}

/* ------------------------------------------------------- causal prefill */

typedef struct {
    double *out, *lse;
    const void *q, *k, *v;
    int dtype;
    const int32_t *cu;
    int B, Hq, Hkv, d;
    double scale;
    volatile int bad;
} prefill_ctx;

static void prefill_item(void *p, long item) {
    prefill_ctx *c = (prefill_ctx *)p;
    int b = (int)(item / c->Hkv), j = (int)(item % c->Hkv);
    long t0 = c->cu[b], n = (long)c->cu[b + 1] - c->cu[b];
    int m = c->Hq / c->Hkv, d = c->d;
    if (n < 0) { c->bad = 1; return; }
    if (n == 0) return;
    double *K = (double *)malloc(sizeof(double) * (size_t)n * d);
    double *V = (double *)malloc(sizeof(double) * (size_t)n * d);
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double *q = (double *)malloc(sizeof(double) * (size_t)d);
    for (long u = 0; u < n; ++u)
        for (int e = 0; e < d; ++e) {
            size_t idx = ((size_t)(t0 + u) * c->Hkv + j) * d + e;
            K[(size_t)u * d + e] = elem(c->k, c->dtype, idx);
            V[(size_t)u * d + e] = elem(c->v, c->dtype, idx);
        }
    for (long t = 0; t < n; ++t)
        for (int i = j * m; i < (j + 1) * m; ++i) {
            size_t row = (size_t)(t0 + t) * c->Hq + i;
            for (int e = 0; e < d; ++e) q[e] = elem(c->q, c->dtype, row * d + e);
            double l = attend(q, K, V, t + 1, d, c->scale, c->out + row * d, s);  /* keys 0..t */
            if (c->lse) c->lse[row] = l;
        }
    free(K); free(V); free(s); free(q);
}

/*
 * Varlen causal prefill.  q [T][Hq][d], k/v [T][Hkv][d] (dtype as the cache
 * dtypes above); cu_seqlens int32 [B+1] with cu[0] = 0, cu[B] = T; out
 * [T][Hq][d] and lse [T][Hq] (may be NULL) in double.  Returns 0 or -1 when
 * cu_seqlens is not non-decreasing.
 */
int oracle_prefill(double *out, double *lse, const void *q, const void *k, const void *v,
                   int dtype, const int32_t *cu_seqlens, int B, int Hq, int Hkv, int d,
                   double scale, int nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return -1;
    for (int b = 0; b < B; ++b)
        if (cu_seqlens[b + 1] < cu_seqlens[b]) return -1;
    prefill_ctx c = {out, lse, q, k, v, dtype, cu_seqlens, B, Hq, Hkv, d, scale, 0};
    run_items(prefill_item, &c, (long)B * Hkv, nthreads);
    return c.bad ? -1 : 0;
}
