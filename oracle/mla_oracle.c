/*
 * CPU oracle for paged MLA decode attention.  TEST INFRASTRUCTURE ONLY: the
 * tests, the smoke check and the benchmark's CPU-baseline leg call it; the
 * library never does.  It shares no code with the CUDA path.
 *
 * What it computes.  The TileLang talk ("Tile级原语与自动推理机制融合，TileAI
 * 社区发起人深度剖析TileLang核心技术与优势", section 什么是「TileLang」) walks
 * through a ~50-line DeepSeek MLA (FlashMLA) decode kernel and its
 * accum_s -> scores_max row-max reduce, but prints neither code nor formula.
 * This file therefore writes out the plain definition of that kernel's
 * result, scaled-dot-product attention of each query row over the latent
 * cache rows it may see:
 *
 *   for batch b, query token i < s_q, head h:
 *     n      = L_b - s_q + 1 + i          (bottom-right causal: the last
 *                                          query token sees all L_b keys)
 *     k_t    = kv[block_table[b][t / 64]][t % 64][0][0:576]   (t < n)
 *     s_t    = scale * sum_{d<576} q[b,i,h,d] * k_t[d]
 *     lse    = log(sum_t exp(s_t))        (natural log, max-subtracted)
 *     out[d] = sum_t exp(s_t - lse) * k_t[d]      for d < 512
 *
 * The values are the first 512 dims of the same cache row (one shared
 * latent head).  An empty row (n <= 0) gives out = 0 and lse = -inf.
 * Everything is evaluated in fp64 from the bf16 input bits; there is no
 * tiling, splitting or reordering beyond the sums written above.
 *
 * oracle_lse_combine writes out the merge of attention results computed over
 * disjoint key sets: lse = log(sum_j exp(lse_j)), out = sum_j
 * exp(lse_j - lse) * out_j.
 *
 * oracle_mla_decode_sparse is the same attention over a selected subset of
 * the cache.  The FlagTree talk write-up ("FlagTree: Triton-TLE 言語拡張、
 * タイルIRバックエンド、およびコンパイラ最適化手法", section 性能テスト)
 * names SparseMLA decode at 128K context but no mechanism; the reading taken
 * is DeepSeek's sparse MLA decode: one query token per batch entry, whose
 * keys are the cache rows at the token positions indices[b][j], j <
 * counts[b] (a list, so a repeated position counts twice), every position
 * in [0, L_b).  With indices[b][j] = j and counts[b] = L_b it is the dense
 * definition above.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define D_QK 576
#define D_V 512
#define PAGE 64

static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t* q;
    const uint16_t* kv;
    int num_pages;
    const int32_t* block_table;
    int max_pages;
    const int32_t* seqlens;
    int batch, s_q, h_q;
    double scale;
    int n_rows;
    const int32_t* rows; /* n_rows x (b, i, h) */
    int key_begin, key_end;
    const int32_t* indices; /* sparse: [batch][topk] token positions, else NULL */
    int topk;
    const int32_t* counts;  /* sparse: keys of each entry */
    double* out;         /* n_rows x 512 */
    double* lse;         /* n_rows */
    int next;            /* shared work counter */
    pthread_mutex_t mu;
    int bad;             /* set when an index is out of range */
} job_t;

/* Cache row of key j of entry b: token j (dense) or indices[b][j] (sparse).
 * NULL when an index is out of range. */
static const uint16_t* key_row(const job_t* J, int b, int j)
{
    int t = j;
    if (J->indices) {
        t = J->indices[(size_t)b * J->topk + j];
        if (t < 0 || t >= J->seqlens[b])
            return NULL;
    }
    if (t / PAGE >= J->max_pages)
        return NULL;
    const int page = J->block_table[(size_t)b * J->max_pages + t / PAGE];
    if (page < 0 || page >= J->num_pages)
        return NULL;
    return J->kv + ((size_t)page * PAGE + (t % PAGE)) * D_QK;
}

/* Attention of one query row over its visible keys restricted to
 * [key_begin, key_end). */
static void one_row(job_t* J, int r, double* s)
{
    const int b = J->rows[3 * r + 0], i = J->rows[3 * r + 1], h = J->rows[3 * r + 2];
    double* o = J->out + (size_t)r * D_V;
    memset(o, 0, sizeof(double) * D_V);
    J->lse[r] = -INFINITY;
    if (b < 0 || b >= J->batch || i < 0 || i >= J->s_q || h < 0 || h >= J->h_q) {
        J->bad = 1;
        return;
    }
    int n;
    if (J->indices) {
        n = J->counts[b];
        if (n < 0 || n > J->topk) {
            J->bad = 1;
            return;
        }
    } else {
        n = J->seqlens[b] - J->s_q + 1 + i;
    }
    int t0 = J->key_begin > 0 ? J->key_begin : 0;
    int t1 = J->key_end < n ? J->key_end : n;
    if (t1 <= t0)
        return;

    const uint16_t* qrow = J->q + (((size_t)b * J->s_q + i) * J->h_q + h) * D_QK;
    double qd[D_QK];
    for (int d = 0; d < D_QK; ++d)
        qd[d] = bf16_to_double(qrow[d]);

    double m = -INFINITY;
    for (int t = t0; t < t1; ++t) {
        const uint16_t* krow = key_row(J, b, t);
        if (!krow) {
            J->bad = 1;
            return;
        }
        double dot = 0.0;
        for (int d = 0; d < D_QK; ++d)
            dot += qd[d] * bf16_to_double(krow[d]);
        s[t - t0] = J->scale * dot;
        if (s[t - t0] > m)
            m = s[t - t0];
    }
    double sum = 0.0;
    for (int t = t0; t < t1; ++t)
        sum += exp(s[t - t0] - m);
    const double lse = m + log(sum);
    for (int t = t0; t < t1; ++t) {
        const double w = exp(s[t - t0] - lse);
        const uint16_t* vrow = key_row(J, b, t);
        for (int d = 0; d < D_V; ++d)
            o[d] += w * bf16_to_double(vrow[d]);
    }
    J->lse[r] = lse;
}

static void* worker(void* arg)
{
    job_t* J = (job_t*)arg;
    int max_n = J->indices ? J->topk : 0;
    for (int b = 0; b < J->batch && !J->indices; ++b)
        if (J->seqlens[b] > max_n)
            max_n = J->seqlens[b];
    double* s = (double*)malloc(sizeof(double) * (size_t)(max_n > 0 ? max_n : 1));
    if (!s) {
        J->bad = 1;
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int r = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (r >= J->n_rows)
            break;
        one_row(J, r, s);
    }
    free(s);
    return NULL;
}

/* Selected rows.  rows = n_rows triples (b, i, h).  Only keys with index in
 * [key_begin, key_end) (and visible) take part; pass 0 and INT32_MAX for the
 * whole sequence.  Returns 0, or -1 on an out-of-range index. */
int oracle_mla_decode_rows(const uint16_t* q, const uint16_t* kv, int num_pages,
                           const int32_t* block_table, int max_pages,
                           const int32_t* cache_seqlens, int batch, int s_q, int h_q,
                           double softmax_scale, int n_rows, const int32_t* rows,
                           int key_begin, int key_end, double* out, double* lse,
                           int nthreads)
{
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q;
    J.kv = kv;
    J.num_pages = num_pages;
    J.block_table = block_table;
    J.max_pages = max_pages;
    J.seqlens = cache_seqlens;
    J.batch = batch;
    J.s_q = s_q;
    J.h_q = h_q;
    J.scale = softmax_scale;
    J.n_rows = n_rows;
    J.rows = rows;
    J.key_begin = key_begin;
    J.key_end = key_end;
    J.out = out;
    J.lse = lse;
    pthread_mutex_init(&J.mu, NULL);
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    pthread_t th[256];
    int started = 0;
    for (int k = 1; k < nthreads; ++k)
        if (pthread_create(&th[started], NULL, worker, &J) == 0)
            ++started;
    worker(&J);
    for (int k = 0; k < started; ++k)
        pthread_join(th[k], NULL);
    pthread_mutex_destroy(&J.mu);
    return J.bad ? -1 : 0;
}

/* Every row.  out is [B, s_q, h_q, 512], lse is [B, h_q, s_q], both fp64. */
int oracle_mla_decode(const uint16_t* q, const uint16_t* kv, int num_pages,
                      const int32_t* block_table, int max_pages, const int32_t* cache_seqlens,
                      int batch, int s_q, int h_q, double softmax_scale, double* out,
                      double* lse, int nthreads)
{
    const int n = batch * s_q * h_q;
    int32_t* rows = (int32_t*)malloc(sizeof(int32_t) * 3 * (size_t)(n > 0 ? n : 1));
    double* l = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (!rows || !l) {
        free(rows);
        free(l);
        return -1;
    }
    int r = 0;
    for (int b = 0; b < batch; ++b)
        for (int i = 0; i < s_q; ++i)
            for (int h = 0; h < h_q; ++h) {
                rows[3 * r] = b;
                rows[3 * r + 1] = i;
                rows[3 * r + 2] = h;
                ++r;
            }
    /* rows are in [B, s_q, h_q] order, which is out's layout */
    int rc = oracle_mla_decode_rows(q, kv, num_pages, block_table, max_pages, cache_seqlens,
                                    batch, s_q, h_q, softmax_scale, n, rows, 0, 0x7fffffff,
                                    out, l, nthreads);
    r = 0;
    for (int b = 0; b < batch; ++b)
        for (int i = 0; i < s_q; ++i)
            for (int h = 0; h < h_q; ++h)
                lse[((size_t)b * h_q + h) * s_q + i] = l[r++];
    free(rows);
    free(l);
    return rc;
}

/* Sparse decode, one query token per entry (s_q = 1), selected rows: rows =
 * n_rows pairs (b, h); key_begin/key_end restrict j (the list position).
 * out [n_rows][512], lse [n_rows].  Returns 0, or -1 on an out-of-range
 * index or count. */
int oracle_mla_decode_sparse_rows(const uint16_t* q, const uint16_t* kv, int num_pages,
                                  const int32_t* block_table, int max_pages,
                                  const int32_t* cache_seqlens, const int32_t* indices, int topk,
                                  const int32_t* counts, int batch, int h_q, double softmax_scale,
                                  int n_rows, const int32_t* rows_bh, int key_begin, int key_end,
                                  double* out, double* lse, int nthreads)
{
    int32_t* rows = (int32_t*)malloc(sizeof(int32_t) * 3 * (size_t)(n_rows > 0 ? n_rows : 1));
    if (!rows)
        return -1;
    for (int r = 0; r < n_rows; ++r) {
        rows[3 * r] = rows_bh[2 * r];
        rows[3 * r + 1] = 0;
        rows[3 * r + 2] = rows_bh[2 * r + 1];
    }
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q;
    J.kv = kv;
    J.num_pages = num_pages;
    J.block_table = block_table;
    J.max_pages = max_pages;
    J.seqlens = cache_seqlens;
    J.batch = batch;
    J.s_q = 1;
    J.h_q = h_q;
    J.scale = softmax_scale;
    J.n_rows = n_rows;
    J.rows = rows;
    J.key_begin = key_begin;
    J.key_end = key_end;
    J.indices = indices;
    J.topk = topk;
    J.counts = counts;
    J.out = out;
    J.lse = lse;
    pthread_mutex_init(&J.mu, NULL);
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    pthread_t th[256];
    int started = 0;
    for (int k = 1; k < nthreads; ++k)
        if (pthread_create(&th[started], NULL, worker, &J) == 0)
            ++started;
    worker(&J);
    for (int k = 0; k < started; ++k)
        pthread_join(th[k], NULL);
    pthread_mutex_destroy(&J.mu);
    free(rows);
    return J.bad ? -1 : 0;
}

/* Merge n results over disjoint key sets. lse_parts [n], o_parts [n][512]. */
void oracle_lse_combine(int n, const double* lse_parts, const double* o_parts, double* lse,
                        double* out)
{
    double m = -INFINITY;
    for (int j = 0; j < n; ++j)
        if (lse_parts[j] > m)
            m = lse_parts[j];
    for (int d = 0; d < D_V; ++d)
        out[d] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double sum = 0.0;
    for (int j = 0; j < n; ++j)
        sum += exp(lse_parts[j] - m);
    *lse = m + log(sum);
    for (int j = 0; j < n; ++j) {
        const double w = exp(lse_parts[j] - *lse);
        for (int d = 0; d < D_V; ++d)
            out[d] += w * o_parts[(size_t)j * D_V + d];
    }
}
