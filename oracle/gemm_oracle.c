/*
 * gemm_oracle.c -- CPU oracle for the dense fp16 GEMM  C = A * B^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this file:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg do.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * What it computes (tilus "A Minimal Hopper Matmul", section "Block Tiling",
 * and its note "Data layout: K-major"):
 *     A is [M, K] and B is [N, K], both row-major with K contiguous;
 *     C is [M, N] with  C[i][j] = sum_{k < K} A[i][k] * B[j][k].
 * The GPU method reaches this exact sum up to rounding order, so the oracle is
 * the definition written out: a plain triple loop, every product and every
 * partial sum in IEEE double, on the same fp16 bits the GPU reads.  Products of
 * two binary16 values are exact in double (11 + 11 significant bits), so the
 * only rounding is in the running double sum.  The result is NOT rounded to
 * fp16; callers compare the GPU's fp16 output against it with a tolerance.
 *
 * Build: plain C99, `gcc -O2 -ffp-contract=off -shared -fPIC -pthread`.
 * -ffp-contract=off keeps each product and each add a separate IEEE rounding on
 * every host (aarch64 would otherwise fuse them), so results match bit for bit
 * across machines and thread counts.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------ */
/* IEEE-754 binary16 -> double, written from the format's definition:
 *   bit 15 sign, bits 14..10 biased exponent (bias 15), bits 9..0 fraction.
 *   exponent 0      : zero / subnormal, value = (-1)^s * 2^-14 * (frac / 1024)
 *   exponent 1..30  : normal,           value = (-1)^s * 2^(e-15) * (1 + frac/1024)
 *   exponent 31     : frac == 0 -> infinity, otherwise NaN                    */
double oracle_half_to_double(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -24);            /* 2^-14 * frac / 2^10 */
    } else if (expo == 31) {
        mag = frac == 0 ? INFINITY : NAN;
    } else {
        mag = ldexp(1024.0 + (double)frac, expo - 25); /* 2^(e-15) * (1024+f)/2^10 */
    }
    return sign ? -mag : mag;
}

/* double -> binary16 bits, round to nearest, ties to even, from the same
 * definition.  Overflow (|x| >= 65520, the midpoint between 65504 and 2^16)
 * gives infinity; NaN gives the quiet NaN 0x7e00.  Used only to state exact
 * closed-form results in fp16 for the bit-exact checks.                     */
uint16_t oracle_double_to_half(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isnan(x)) return 0x7e00u;
    if (a == 0.0) return sign;
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u);

    int e;                          /* a = m * 2^e with m in [0.5, 1) */
    (void)frexp(a, &e);
    int unbiased = e - 1;           /* a = 1.xxx * 2^unbiased */
    if (unbiased < -14) unbiased = -14;   /* subnormal range shares 2^-24 spacing */
    /* quantum (spacing of representable values) in this binade */
    double scaled = ldexp(a, 10 - unbiased);   /* a / 2^(unbiased-10) */
    double fl = floor(scaled);
    double rem = scaled - fl;                  /* exact: scaled has < 53 bits */
    double q = fl;
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) q = fl + 1.0;
    /* q in [0, 2048]; 2048 means carry into the next binade */
    if (q >= 2048.0) { q = 1024.0; unbiased += 1; }
    if (unbiased > 15) return (uint16_t)(sign | 0x7c00u);
    uint16_t bits;
    if (q < 1024.0) {
        /* only reachable for unbiased == -14: subnormal, exponent field 0 */
        bits = (uint16_t)q;
    } else {
        bits = (uint16_t)(((unbiased + 15) << 10) | ((int)q - 1024));
    }
    return (uint16_t)(sign | bits);
}

void oracle_decode_f16(const uint16_t* h, double* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_half_to_double(h[i]);
}

void oracle_encode_f16(const double* x, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_double_to_half(x[i]);
}

/* ------------------------------------------------------------------------ */
/* One output element: the K-long dot product of row i of A and row j of B,
 * both K-contiguous (the B^T convention), summed in order k = 0 .. K-1.      */
static double dot_row_row(const double* lut, const uint16_t* a_row,
                          const uint16_t* b_row, int64_t K)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double p = lut[a_row[k]] * lut[b_row[k]];
        acc = acc + p;
    }
    return acc;
}

/* A 65536-entry decode table built from oracle_half_to_double, so the inner
 * loop is a lookup instead of a decode.  Built once, read-only afterwards.  */
static double g_lut[65536];
static pthread_once_t g_lut_once = PTHREAD_ONCE_INIT;
static void build_lut(void)
{
    for (int h = 0; h < 65536; ++h) g_lut[h] = oracle_half_to_double((uint16_t)h);
}

typedef struct {
    const uint16_t* A; const uint16_t* B;
    int64_t M, N, K;
    /* mode 0: full C[M,N]; 1: listed rows -> out[r*N + j];
       2: listed cols -> out[c*M + i] */
    int mode;
    const int64_t* idx; int64_t nidx;
    double* out;
    int64_t begin, end;     /* range of the outer index this worker owns */
} job_t;

static void* worker(void* p)
{
    job_t* jb = (job_t*)p;
    const int64_t N = jb->N, K = jb->K, M = jb->M;
    for (int64_t u = jb->begin; u < jb->end; ++u) {
        if (jb->mode == 0) {
            const uint16_t* a_row = jb->A + u * K;
            for (int64_t j = 0; j < N; ++j)
                jb->out[u * N + j] = dot_row_row(g_lut, a_row, jb->B + j * K, K);
        } else if (jb->mode == 1) {
            const uint16_t* a_row = jb->A + jb->idx[u] * K;
            for (int64_t j = 0; j < N; ++j)
                jb->out[u * N + j] = dot_row_row(g_lut, a_row, jb->B + j * K, K);
        } else {
            const uint16_t* b_row = jb->B + jb->idx[u] * K;
            for (int64_t i = 0; i < M; ++i)
                jb->out[u * M + i] = dot_row_row(g_lut, jb->A + i * K, b_row, K);
        }
    }
    return NULL;
}

static int resolve_threads(int threads)
{
    if (threads > 0) return threads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static int run_jobs(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N,
                    int64_t K, int mode, const int64_t* idx, int64_t nidx,
                    double* out, int threads)
{
    pthread_once(&g_lut_once, build_lut);
    const int64_t outer = mode == 0 ? M : nidx;
    int T = resolve_threads(threads);
    if ((int64_t)T > outer) T = outer > 0 ? (int)outer : 1;
    job_t* jobs = (job_t*)calloc((size_t)T, sizeof(job_t));
    pthread_t* tid = (pthread_t*)calloc((size_t)T, sizeof(pthread_t));
    if (!jobs || !tid) { free(jobs); free(tid); return -1; }
    for (int t = 0; t < T; ++t) {
        jobs[t] = (job_t){A, B, M, N, K, mode, idx, nidx, out,
                          outer * t / T, outer * (t + 1) / T};
    }
    int spawned = 0;
    for (int t = 1; t < T; ++t)
        if (pthread_create(&tid[t], NULL, worker, &jobs[t]) == 0) ++spawned;
        else { worker(&jobs[t]); tid[t] = 0; }
    worker(&jobs[0]);
    for (int t = 1; t < T; ++t) if (tid[t]) pthread_join(tid[t], NULL);
    (void)spawned;
    free(jobs); free(tid);
    return T;
}

/* Full product: C[i*N + j] for all i < M, j < N.  Returns threads used.    */
int oracle_gemm_f64(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N,
                    int64_t K, double* C, int threads)
{
    return run_jobs(A, B, M, N, K, 0, NULL, 0, C, threads);
}

/* Selected rows: out[r*N + j] = C[rows[r]][j].  Returns threads used.       */
int oracle_gemm_rows_f64(const uint16_t* A, const uint16_t* B, int64_t M,
                         int64_t N, int64_t K, const int64_t* rows,
                         int64_t nrows, double* out, int threads)
{
    return run_jobs(A, B, M, N, K, 1, rows, nrows, out, threads);
}

/* Selected columns: out[c*M + i] = C[i][cols[c]].  Returns threads used.    */
int oracle_gemm_cols_f64(const uint16_t* A, const uint16_t* B, int64_t M,
                         int64_t N, int64_t K, const int64_t* cols,
                         int64_t ncols, double* out, int threads)
{
    return run_jobs(A, B, M, N, K, 2, cols, ncols, out, threads);
}
