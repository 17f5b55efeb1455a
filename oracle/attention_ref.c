/*
 * Plain fp64 CPU oracle for causal multi-head attention — TEST INFRASTRUCTURE.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this file's library.  It shares no code, header or constant with the
 * CUDA path; its only input is the float32 arrays the seeded generators make.
 *
 * What it computes is the definition on the page "Hand-written masked
 * multi-head attention CUDA kernel: underlying logic and practice"
 * (xdnf.cn/news/357253), section 2:
 *
 *     A = softmax(Q K^T / sqrt(d_k) + M),  M = 0 on/below the diagonal,
 *                                          M = -inf above it,
 *     O = A V
 *
 * (the page writes the last product as "A V^T"; only A V has matching
 * dimensions, so that is the reading taken).  Section 2.2 of the same page
 * fixes the mask: query row i may use key j only when j <= i.  Section 2.3
 * gives the max subtraction, which is exact here because softmax is
 * unchanged when a constant is subtracted from a whole row; the page's clamp
 * of the maximum to +-15 is an fp16 device and is not applied.  The scale is
 * an argument (1/sqrt(D) in every workload); it multiplies the dot product
 * before the mask is applied.
 *
 * Besides O, each row reports LSE = ln(sum_{valid j} exp(scale * q_i . k_j)),
 * the natural log of the softmax denominator, written as m + ln(Z) with m the
 * row maximum.
 *
 * Key padding (optional): with per-sequence key lengths L_b, key j of
 * sequence b exists only when j < L_b, the padded scores being -inf (page
 * "Week 4 CUDA notes" section 2.2 sets padded positions to -inf before the
 * softmax).  A row with no valid key has O = 0 and LSE = -inf.
 *
 * Everything is evaluated in double: float inputs are widened exactly, every
 * product and sum is double, nothing is rounded back.  No blocking, fusion or
 * reordering: each row is one pass over its valid keys to get the scores,
 * one for the maximum, one for the weights and their sum, one for the
 * weighted sum of V rows.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* One output row of prefill attention.
 * q: D doubles-worth of query (float), K,V: S x D rows of one (b,h) slice.
 * n_valid: number of keys the row may see (keys 0..n_valid-1).
 * s: scratch of at least n_valid doubles. */
static void attention_row(const float *q, const float *K, const float *V,
                          int64_t n_valid, int64_t D, double scale,
                          double *s, double *o, double *lse)
{
    if (n_valid == 0) { /* no valid key: empty sum */
        for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
        *lse = -INFINITY;
        return;
    }
    /* scores s_j = scale * sum_d q_d k_jd  (page 3, section 2: QK^T/sqrt(d_k)) */
    for (int64_t j = 0; j < n_valid; ++j) {
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d)
            dot += (double)q[d] * (double)K[j * D + d];
        s[j] = scale * dot;
    }
    /* row maximum (page 3, section 2.3: subtract the max before exp) */
    double m = -INFINITY;
    for (int64_t j = 0; j < n_valid; ++j)
        if (s[j] > m) m = s[j];
    /* weights w_j = exp(s_j - m) and their sum Z */
    double Z = 0.0;
    for (int64_t j = 0; j < n_valid; ++j) {
        s[j] = exp(s[j] - m);
        Z += s[j];
    }
    /* O = sum_j (w_j / Z) V_j  (the product A V) */
    for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
    for (int64_t j = 0; j < n_valid; ++j) {
        double a = s[j] / Z;
        for (int64_t d = 0; d < D; ++d)
            o[d] += a * (double)V[j * D + d];
    }
    *lse = m + log(Z);
}

typedef struct {
    const float *Q, *K, *V;
    int64_t B, H, S, D;
    double scale;
    int causal;
    const int64_t *rows; /* flat ids (b*H+h)*S+i, or NULL for all rows */
    int64_t nrows;
    double *O, *LSE;
    int tid, nthreads;
    int status;
    const int32_t *key_lens; /* [B] key lengths, or NULL: every sequence has S keys */
} prefill_job;

static void *prefill_worker(void *arg)
{
    prefill_job *jb = (prefill_job *)arg;
    double *s = (double *)malloc((size_t)(jb->S > 0 ? jb->S : 1) * sizeof(double));
    if (!s) { jb->status = 1; return NULL; }
    /* rows are dealt round-robin so causal rows of every length mix evenly */
    for (int64_t r = jb->tid; r < jb->nrows; r += jb->nthreads) {
        int64_t flat = jb->rows ? jb->rows[r] : r;
        int64_t bh = flat / jb->S, i = flat % jb->S;
        const float *base_q = jb->Q + (bh * jb->S + i) * jb->D;
        const float *base_k = jb->K + bh * jb->S * jb->D;
        const float *base_v = jb->V + bh * jb->S * jb->D;
        int64_t n_valid = jb->causal ? i + 1 : jb->S; /* keys j <= i (page 3, 2.2) */
        if (jb->key_lens) { /* and j < L_b: both bounds keep a prefix of the keys */
            int64_t L = jb->key_lens[bh / jb->H];
            if (n_valid > L) n_valid = L;
        }
        attention_row(base_q, base_k, base_v, n_valid, jb->D, jb->scale, s,
                      jb->O + r * jb->D, jb->LSE + r);
    }
    free(s);
    return NULL;
}

static int resolve_threads(int nthreads)
{
    if (nthreads > 0) return nthreads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Prefill oracle.  Q, K, V: float32 [B, H, S, D] contiguous.
 * key_lens: int32 [B], each in [0, S], or NULL (every sequence has S keys).
 * rows == NULL: every row, O is [B*H*S, D], LSE is [B*H*S].
 * rows != NULL: nrows flat row ids (b*H + h)*S + i; O is [nrows, D] and LSE
 * [nrows], in the order given.  Returns 0 on success, the number of threads
 * actually used is written to *threads_used when it is not NULL.
 */
int oracle_attention_rows_kl(const float *Q, const float *K, const float *V,
                             int64_t B, int64_t H, int64_t S, int64_t D,
                             double scale, int causal, const int32_t *key_lens,
                             const int64_t *rows, int64_t nrows,
                             double *O, double *LSE, int nthreads, int *threads_used)
{
    if (B < 0 || H < 0 || S < 0 || D < 1) return 2;
    if (key_lens)
        for (int64_t b = 0; b < B; ++b)
            if (key_lens[b] < 0 || key_lens[b] > S) return 2;
    if (!rows) nrows = B * H * S;
    if (rows)
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= B * H * S) return 2;
    int nt = resolve_threads(nthreads);
    if ((int64_t)nt > nrows) nt = nrows > 0 ? (int)nrows : 1;
    if (threads_used) *threads_used = nt;
    prefill_job *jobs = (prefill_job *)calloc((size_t)nt, sizeof(prefill_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return 1; }
    for (int t = 0; t < nt; ++t) {
        prefill_job j = {Q, K, V, B, H, S, D, scale, causal, rows, nrows, O, LSE, t, nt, 0, key_lens};
        jobs[t] = j;
    }
    for (int t = 1; t < nt; ++t) pthread_create(&th[t], NULL, prefill_worker, &jobs[t]);
    prefill_worker(&jobs[0]);
    int status = jobs[0].status;
    for (int t = 1; t < nt; ++t) {
        pthread_join(th[t], NULL);
        if (jobs[t].status) status = jobs[t].status;
    }
    free(jobs);
    free(th);
    return status;
}

/* The same without key padding. */
int oracle_attention_rows(const float *Q, const float *K, const float *V,
                          int64_t B, int64_t H, int64_t S, int64_t D,
                          double scale, int causal,
                          const int64_t *rows, int64_t nrows,
                          double *O, double *LSE, int nthreads, int *threads_used)
{
    return oracle_attention_rows_kl(Q, K, V, B, H, S, D, scale, causal, NULL, rows, nrows,
                                    O, LSE, nthreads, threads_used);
}

/*
 * Single-query decode oracle (the page's "mmha" case: one new query per
 * sequence attends to every cached key of its own sequence, so no key lies
 * above the diagonal and the mask removes nothing).
 *
 * q: float32 [B, H, D].  Kc, Vc: float32 [sum_b seqlens[b], H, D], the
 * sequences packed one after another in batch order.  O: [B, H, D],
 * LSE: [B, H].  A sequence of length 0 gives O = 0 and LSE = -inf.
 */
typedef struct {
    const float *q, *Kc, *Vc;
    const int32_t *seqlens;
    const int64_t *offs;
    int64_t B, H, D;
    double scale;
    double *O, *LSE;
    int tid, nthreads;
    int64_t max_len;
    int status;
} decode_job;

static void *decode_worker(void *arg)
{
    decode_job *jb = (decode_job *)arg;
    int64_t D = jb->D, H = jb->H;
    double *s = (double *)malloc((size_t)(jb->max_len > 0 ? jb->max_len : 1) * sizeof(double));
    float *k = (float *)malloc((size_t)(jb->max_len > 0 ? jb->max_len : 1) * (size_t)D * sizeof(float));
    float *v = (float *)malloc((size_t)(jb->max_len > 0 ? jb->max_len : 1) * (size_t)D * sizeof(float));
    if (!s || !k || !v) { jb->status = 1; free(s); free(k); free(v); return NULL; }
    for (int64_t bh = jb->tid; bh < jb->B * H; bh += jb->nthreads) {
        int64_t b = bh / H, h = bh % H;
        int64_t L = jb->seqlens[b];
        double *o = jb->O + bh * D;
        if (L == 0) {
            for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
            jb->LSE[bh] = -INFINITY;
            continue;
        }
        /* gather this head's rows of the packed cache into [L, D] */
        for (int64_t t = 0; t < L; ++t) {
            memcpy(k + t * D, jb->Kc + ((jb->offs[b] + t) * H + h) * D, (size_t)D * sizeof(float));
            memcpy(v + t * D, jb->Vc + ((jb->offs[b] + t) * H + h) * D, (size_t)D * sizeof(float));
        }
        attention_row(jb->q + bh * D, k, v, L, D, jb->scale, s, o, jb->LSE + bh);
    }
    free(s); free(k); free(v);
    return NULL;
}

int oracle_decode(const float *q, const float *Kc, const float *Vc, const int32_t *seqlens,
                  int64_t B, int64_t H, int64_t D, double scale,
                  double *O, double *LSE, int nthreads, int *threads_used)
{
    if (B < 0 || H < 0 || D < 1) return 2;
    int64_t *offs = (int64_t *)calloc((size_t)(B > 0 ? B : 1), sizeof(int64_t));
    if (!offs) return 1;
    int64_t acc = 0, max_len = 0;
    for (int64_t b = 0; b < B; ++b) {
        if (seqlens[b] < 0) { free(offs); return 2; }
        offs[b] = acc;
        acc += seqlens[b];
        if (seqlens[b] > max_len) max_len = seqlens[b];
    }
    int nt = resolve_threads(nthreads);
    if ((int64_t)nt > B * H) nt = B * H > 0 ? (int)(B * H) : 1;
    if (threads_used) *threads_used = nt;
    decode_job *jobs = (decode_job *)calloc((size_t)nt, sizeof(decode_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); free(offs); return 1; }
    for (int t = 0; t < nt; ++t) {
        decode_job j = {q, Kc, Vc, seqlens, offs, B, H, D, scale, O, LSE, t, nt, max_len, 0};
        jobs[t] = j;
    }
    for (int t = 1; t < nt; ++t) pthread_create(&th[t], NULL, decode_worker, &jobs[t]);
    decode_worker(&jobs[0]);
    int status = jobs[0].status;
    for (int t = 1; t < nt; ++t) {
        pthread_join(th[t], NULL);
        if (jobs[t].status) status = jobs[t].status;
    }
    free(jobs); free(th); free(offs);
    return status;
}
