/*
 * Oracle for the fused GEMM  C = act(A·B + bias)  — plain fp64 CPU code.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library includes, links or
 * calls this file; only the test-suite, the smoke check and the CPU-baseline leg
 * of the benchmark load it (through oracle/gemm.py).
 *
 * What it follows:
 *   - "Tile Selection: Cost Models Against Measurement", section "The structure of
 *     the search space": C = AB with C of shape M x N and reduction depth K.
 *   - "Tiling the hierarchy", fusion section: the bias + activation epilogue is an
 *     elementwise chain applied to the GEMM output.
 * The pages do not say what "bias" is nor which GELU; the readings taken here are
 * bias[n] broadcast over rows and the exact (erf) GELU, 0.5·x·(1 + erf(x/√2)).
 *
 * Everything is computed in double precision from inputs that are already the
 * rounded values the device sees (bf16 values are exact in float, so every input
 * arrives here as float).  The sum runs over k in increasing order for each
 * (m, n); there is no blocking and no reordering beyond the m-k-n loop nest.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Epilogue codes: 0 = none, 1 = + bias, 2 = relu(. + bias), 3 = gelu(. + bias). */
static double oracle_epilogue(double x, double b, int epi)
{
    if (epi == 0) return x;
    x += b;
    if (epi == 2) return x > 0.0 ? x : 0.0;
    if (epi == 3) return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
    return x;
}

typedef struct {
    const float *A, *B, *bias;
    double *C;
    int64_t M, N, K, m_begin, m_end;
    int epi;
    double alpha;
} oracle_rows_job;

static void *oracle_rows_worker(void *arg)
{
    const oracle_rows_job *j = (const oracle_rows_job *)arg;
    for (int64_t m = j->m_begin; m < j->m_end; ++m) {
        double *crow = j->C + m * j->N;
        for (int64_t n = 0; n < j->N; ++n) crow[n] = 0.0;
        for (int64_t k = 0; k < j->K; ++k) {
            const double a = (double)j->A[m * j->K + k];
            const float *brow = j->B + k * j->N;
            for (int64_t n = 0; n < j->N; ++n) crow[n] += a * (double)brow[n];
        }
        for (int64_t n = 0; n < j->N; ++n)
            crow[n] = oracle_epilogue(j->alpha * crow[n], j->bias ? (double)j->bias[n] : 0.0, j->epi);
    }
    return NULL;
}

/* Full product: C[m*N + n] = act(alpha · sum_k A[m*K+k]·B[k*N+n] + bias[n]),
 * rows split into contiguous blocks over `threads` POSIX threads (threads <= 1:
 * caller's thread only).  alpha is the product's scale (the tensor scales of
 * FP8 operands; 1 otherwise).  Returns 0, or -1 on bad arguments. */
int oracle_gemm(const float *A, const float *B, const float *bias, int epi, double alpha,
                int64_t M, int64_t N, int64_t K, double *C, int threads)
{
    if (M < 0 || N < 0 || K < 0 || epi < 0 || epi > 3) return -1;
    if (epi != 0 && bias == NULL && N > 0) return -1;
    if (M == 0 || N == 0) return 0;
    if (threads < 1) threads = 1;
    if (threads > M) threads = (int)M;
    oracle_rows_job *jobs = (oracle_rows_job *)calloc((size_t)threads, sizeof(*jobs));
    pthread_t *tids = (pthread_t *)calloc((size_t)threads, sizeof(*tids));
    if (!jobs || !tids) { free(jobs); free(tids); return -1; }
    for (int t = 0; t < threads; ++t) {
        jobs[t].A = A; jobs[t].B = B; jobs[t].bias = bias; jobs[t].C = C;
        jobs[t].M = M; jobs[t].N = N; jobs[t].K = K; jobs[t].epi = epi; jobs[t].alpha = alpha;
        jobs[t].m_begin = (M * t) / threads;
        jobs[t].m_end = (M * (t + 1)) / threads;
    }
    int started = 0;
    for (int t = 1; t < threads; ++t) {
        if (pthread_create(&tids[t], NULL, oracle_rows_worker, &jobs[t]) != 0) break;
        started = t;
    }
    oracle_rows_worker(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    /* rows of threads that could not be started run here */
    for (int t = started + 1; t < threads; ++t) oracle_rows_worker(&jobs[t]);
    free(jobs); free(tids);
    return 0;
}

/* Selected entries, one dot product each: out[i] = C[rows[i], cols[i]].  Used to
 * check full-size runs whose whole product would take too long here. */
int oracle_gemm_entries(const float *A, const float *B, const float *bias, int epi, double alpha,
                        int64_t M, int64_t N, int64_t K,
                        const int64_t *rows, const int64_t *cols, int64_t count, double *out)
{
    if (epi < 0 || epi > 3) return -1;
    for (int64_t i = 0; i < count; ++i) {
        const int64_t m = rows[i], n = cols[i];
        if (m < 0 || m >= M || n < 0 || n >= N) return -1;
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k) s += (double)A[m * K + k] * (double)B[k * N + n];
        out[i] = oracle_epilogue(alpha * s, bias ? (double)bias[n] : 0.0, epi);
    }
    return 0;
}

/* Round-to-nearest-even of a double to bfloat16 (8 significant bits, exponent
 * range of float), returned as the 16-bit pattern.  Written from the definition:
 * scale the significand to an integer with 8 bits, round half to even, scale back. */
static uint16_t oracle_bf16_bits(double x)
{
    float f;
    uint32_t u;
    if (isnan(x)) return 0x7FC0;
    if (x == 0.0 || isinf(x)) {
        f = (float)x;
        memcpy(&u, &f, 4);
        return (uint16_t)(u >> 16);
    }
    int e;
    double frac = frexp(fabs(x), &e);               /* |x| = frac·2^e, frac in [0.5, 1) */
    int q = e - 8;                                   /* quantum exponent for 8 bits */
    if (q < -133) q = -133;                          /* bf16 subnormal quantum 2^-133 */
    double scaled = ldexp(fabs(x), -q);
    double r = nearbyint(scaled);                    /* default mode: nearest, ties to even */
    double y = ldexp(r, q);
    if (y >= 0x1.0p128) y = INFINITY;                /* overflow past the largest bf16 */
    (void)frac;
    f = (float)(x < 0 ? -y : y);
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

void oracle_round_bf16(const double *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_bits(x[i]);
}

/* Round a double to the nearest float (ties to even) — the fp32 output path. */
void oracle_round_f32(const double *x, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (float)x[i];
}
