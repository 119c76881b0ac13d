/*
 * CPU oracle for the tensor-core GEMM.  TEST INFRASTRUCTURE ONLY: the tests
 * and the benchmark's CPU-baseline leg call it; the library never does.  It
 * shares no code with the CUDA path.
 *
 * The GEMM tutorial summary ("Designing high-performance GPU kernels with
 * TileLang: Tensor-Core GEMM", its comparison table) measures an FP16
 * 2048 x 2048 x 2048 matrix product against cuBLAS, with a relative error
 * under 2e-2.  The definition written out here:
 *     C[m][n] = sum_{k < K} A[m][k] * B[k][n]
 * A row-major [M][K], B row-major [K][N], evaluated in fp64 from the fp16
 * (or bf16) input bits, as a plain loop over k.
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

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits; exponent 0 holds zero and the subnormals, 31 infinity and NaN. */
static double f16_value(uint16_t bits)
{
    const int sign = (bits >> 15) & 1;
    const int e = (bits >> 10) & 0x1f;
    const int f = bits & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* f / 2^10 * 2^-14 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1.0 + (double)f / 1024.0, e - 15);
    return sign ? -v : v;
}

/* One entry of C = A B; fmt 0 = fp16 inputs, 1 = bf16 inputs. */
static double gemm_entry(const uint16_t* A, const uint16_t* B, int N, int K, int fmt, int m,
                         int n)
{
    double acc = 0.0;
    for (int k = 0; k < K; ++k) {
        const uint16_t a = A[(size_t)m * K + k], b = B[(size_t)k * N + n];
        acc += fmt ? bf16_value(a) * bf16_value(b) : f16_value(a) * f16_value(b);
    }
    return acc;
}

typedef struct {
    const uint16_t* A;
    const uint16_t* B;
    int M, N, K, fmt;
    int n_entries;           /* -1: all of C, row by row */
    const int32_t* entries;  /* n_entries x (m, n) */
    double* out;
    int next;
    pthread_mutex_t mu;
} gemm_job_t;

static void* gemm_worker(void* arg)
{
    gemm_job_t* J = (gemm_job_t*)arg;
    const int total = J->n_entries < 0 ? J->M : J->n_entries;
    const int chunk = J->n_entries < 0 ? 1 : 64;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        const int w0 = J->next;
        J->next += chunk;
        pthread_mutex_unlock(&J->mu);
        if (w0 >= total)
            break;
        const int w1 = w0 + chunk < total ? w0 + chunk : total;
        for (int w = w0; w < w1; ++w) {
            if (J->n_entries < 0) {
                for (int n = 0; n < J->N; ++n)
                    J->out[(size_t)w * J->N + n] = gemm_entry(J->A, J->B, J->N, J->K, J->fmt, w, n);
            } else {
                const int m = J->entries[2 * w], n = J->entries[2 * w + 1];
                J->out[w] = gemm_entry(J->A, J->B, J->N, J->K, J->fmt, m, n);
            }
        }
    }
    return NULL;
}

static int run_gemm(gemm_job_t* J, int nthreads)
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
        if (pthread_create(&th[t], NULL, gemm_worker, J) == 0)
            ++started;
    if (started == 0)
        gemm_worker(J);
    for (int t = 0; t < started; ++t)
        pthread_join(th[t], NULL);
    pthread_mutex_destroy(&J->mu);
    return 0;
}

/* All of C [M][N] (fp64). */
int oracle_gemm(const uint16_t* A, const uint16_t* B, int M, int N, int K, int fmt, double* C,
                int nthreads)
{
    gemm_job_t J = {A, B, M, N, K, fmt, -1, NULL, C, 0};
    return run_gemm(&J, nthreads);
}

/* Selected entries: entries = n x (m, n) -> out[n]. */
int oracle_gemm_entries(const uint16_t* A, const uint16_t* B, int M, int N, int K, int fmt,
                        int n, const int32_t* entries, double* out, int nthreads)
{
    for (int j = 0; j < n; ++j)
        if (entries[2 * j] < 0 || entries[2 * j] >= M || entries[2 * j + 1] < 0 ||
            entries[2 * j + 1] >= N)
            return -1;
    gemm_job_t J = {A, B, M, N, K, fmt, n, entries, out, 0};
    return run_gemm(&J, nthreads);
}
