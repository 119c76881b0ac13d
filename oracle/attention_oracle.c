/*
 * CPU oracle for dense (FlashAttention-style) attention forward.  TEST
 * INFRASTRUCTURE ONLY: the tests and the benchmark's CPU-baseline leg call
 * it; the library never does.  It shares no code with the CUDA path.
 *
 * The pages name FlashAttention twice without a formula: the TileLang talk
 * ("Tile级原语与自动推理机制融合，TileAI社区发起人深度剖析TileLang核心技术与优势",
 * its performance section) reports MLA, FlashAttention and block-sparse
 * kernels on par with CUTLASS, and the GEMM tutorial summary ("Designing
 * high-performance GPU kernels with TileLang: Tensor-Core GEMM", key
 * capabilities) lists FlashAttention and fused GEMM + softmax, which keep the
 * score matrix out of HBM.  What such a kernel computes is plain
 * scaled-dot-product attention, written out here:
 *
 *   for batch b, head h, query i < S:
 *     keys t visible: t <= i (causal, query i at position i) or all t < S
 *     s_t    = scale * sum_{d < d_qk} q[b][i][h][d] * k[b][t][h][d]
 *     lse    = log(sum_t exp(s_t))          (natural log, max-subtracted)
 *     out[d] = sum_t exp(s_t - lse) * v[b][t][h][d]    for d < d_v
 *
 * Layouts: q, k [B][S][H][d_qk], v [B][S][H][d_v] (bf16 bits), out
 * [B][S][H][d_v] and lse [B][H][S] in fp64.  Every sum is a plain loop in the
 * order written, in fp64 from the bf16 inputs.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_value(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q, *k, *v;
    int B, S, H, dqk, dv, causal;
    double scale;
    int n_rows;              /* -1: every (b, h, i); else rows = n x (b, h, i) */
    const int32_t* rows;
    double *out, *lse;       /* [n][d_v], [n] for a row list; full layouts otherwise */
    int next;
    pthread_mutex_t mu;
} att_job_t;

static void one_row(const att_job_t* J, int b, int h, int i, double* o, double* lse_out)
{
    const int n = J->causal ? i + 1 : J->S;
    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    const uint16_t* q = J->q + (((size_t)b * J->S + i) * J->H + h) * J->dqk;
    double m = -INFINITY;
    for (int t = 0; t < n; ++t) {
        const uint16_t* k = J->k + (((size_t)b * J->S + t) * J->H + h) * J->dqk;
        double dot = 0.0;
        for (int d = 0; d < J->dqk; ++d)
            dot += bf16_value(q[d]) * bf16_value(k[d]);
        s[t] = J->scale * dot;
        if (s[t] > m)
            m = s[t];
    }
    double sum = 0.0;
    for (int t = 0; t < n; ++t)
        sum += exp(s[t] - m);
    const double lse = m + log(sum);
    for (int d = 0; d < J->dv; ++d)
        o[d] = 0.0;
    for (int t = 0; t < n; ++t) {
        const double w = exp(s[t] - lse);
        const uint16_t* v = J->v + (((size_t)b * J->S + t) * J->H + h) * J->dv;
        for (int d = 0; d < J->dv; ++d)
            o[d] += w * bf16_value(v[d]);
    }
    *lse_out = lse;
    free(s);
}

static void* att_worker(void* arg)
{
    att_job_t* J = (att_job_t*)arg;
    const int total = J->n_rows < 0 ? J->B * J->H * J->S : J->n_rows;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        const int w = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (w >= total)
            break;
        int b, h, i;
        double *o, *l;
        if (J->n_rows < 0) {
            b = w / (J->H * J->S);
            h = (w / J->S) % J->H;
            i = w % J->S;
            o = J->out + (((size_t)b * J->S + i) * J->H + h) * J->dv;
            l = J->lse + ((size_t)b * J->H + h) * J->S + i;
        } else {
            b = J->rows[3 * w];
            h = J->rows[3 * w + 1];
            i = J->rows[3 * w + 2];
            o = J->out + (size_t)w * J->dv;
            l = J->lse + w;
        }
        one_row(J, b, h, i, o, l);
    }
    return NULL;
}

static int run(att_job_t* J, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    pthread_t th[256];
    pthread_mutex_init(&J->mu, NULL);
    J->next = 0;
    int started = 0;
    for (int t = 0; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, att_worker, J) == 0)
            ++started;
    if (started == 0)
        att_worker(J);
    for (int t = 0; t < started; ++t)
        pthread_join(th[t], NULL);
    pthread_mutex_destroy(&J->mu);
    return 0;
}

/* Every row: out [B][S][H][d_v], lse [B][H][S]. */
int oracle_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, int B, int S,
                     int H, int dqk, int dv, int causal, double scale, double* out, double* lse,
                     int nthreads)
{
    att_job_t J = {q, k, v, B, S, H, dqk, dv, causal, scale, -1, NULL, out, lse, 0};
    return run(&J, nthreads);
}

/* Selected rows: rows = n x (b, h, i) -> out [n][d_v], lse [n]. */
int oracle_attention_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v, int B, int S,
                          int H, int dqk, int dv, int causal, double scale, int n,
                          const int32_t* rows, double* out, double* lse, int nthreads)
{
    for (int r = 0; r < n; ++r)
        if (rows[3 * r] < 0 || rows[3 * r] >= B || rows[3 * r + 1] < 0 || rows[3 * r + 1] >= H ||
            rows[3 * r + 2] < 0 || rows[3 * r + 2] >= S)
            return -1;
    att_job_t J = {q, k, v, B, S, H, dqk, dv, causal, scale, n, rows, out, lse, 0};
    return run(&J, nthreads);
}
