/*
 * Oracle for the bf16 GEMM  C[M,N] = A[M,K] . B[N,K]^T  -- TEST INFRASTRUCTURE ONLY.
 *
 * This file is the plain, slow, obviously correct definition the CUDA library is
 * checked against.  Only the tests, the smoke check and the bench's CPU-baseline
 * leg may load it; the library never does, and this file shares no code with it.
 *
 * What it computes (the definition, written out):
 *
 *     ref[m][n] = sum_{k = 0}^{K-1}  double(A[m][k]) * double(B[n][k])
 *
 * with A[m][k] = A[m*lda + k] and B[n][k] = B[n*ldb + k] stored as bf16 bit
 * patterns, each decoded exactly to fp64, the products formed in fp64 and summed
 * in fp64 in increasing k.  The result is NOT rounded to bf16.  This follows the
 * pages' rule that a kernel is checked against a CPU double-precision version
 * before it is timed (spark-kernels, "how things are measured") and that GEMM
 * references are fp64 (UwULLM kernel-dev, section 6 "Numerics rules").
 *
 * The sampled mode evaluates the same sum for the intersections of chosen rows
 * and columns only, as the gemm3 benchmarks page does for its 128 x 128 sampled
 * check ("Correctness").  Threads split the output rows; they never change the
 * arithmetic of any one element.
 */
#include <pthread.h>
#include <stdint.h>
#include <string.h>

/* bf16 is the top half of an IEEE-754 binary32: widen by 16 zero bits. */
static double bf16_to_f64(uint16_t h)
{
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* One output element: the fp64 sum over k in increasing order. */
static double dot_row_col(const uint16_t *a_row, const uint16_t *b_row, int64_t K)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k)
        acc += bf16_to_f64(a_row[k]) * bf16_to_f64(b_row[k]);
    return acc;
}

typedef struct {
    const uint16_t *A, *B;
    double *C;
    int64_t N, K, lda, ldb, ldc;
    const int64_t *rows; /* rows of C to compute (full mode: 0..M-1)          */
    int64_t nrows;
    const int64_t *cols; /* NULL: all N columns; else the sampled columns      */
    int64_t ncols;
    int tid, nthreads;
} oracle_job;

static void *oracle_worker(void *p)
{
    const oracle_job *j = (const oracle_job *)p;
    for (int64_t i = j->tid; i < j->nrows; i += j->nthreads) {
        const int64_t m = j->rows ? j->rows[i] : i;
        const uint16_t *a_row = j->A + m * j->lda;
        if (j->cols == NULL) {
            for (int64_t n = 0; n < j->N; ++n)
                j->C[i * j->ldc + n] = dot_row_col(a_row, j->B + n * j->ldb, j->K);
        } else {
            for (int64_t c = 0; c < j->ncols; ++c)
                j->C[i * j->ldc + c] = dot_row_col(a_row, j->B + j->cols[c] * j->ldb, j->K);
        }
    }
    return NULL;
}

static int run_jobs(oracle_job base, int nthreads)
{
    enum { MAX_THREADS = 256 };
    pthread_t th[MAX_THREADS];
    oracle_job jobs[MAX_THREADS];
    if (nthreads < 1) nthreads = 1;
    if (nthreads > MAX_THREADS) nthreads = MAX_THREADS;
    if ((int64_t)nthreads > base.nrows && base.nrows > 0) nthreads = (int)base.nrows;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].tid = t;
        jobs[t].nthreads = nthreads;
        if (t == 0) continue; /* the calling thread takes share 0 */
        if (pthread_create(&th[t], NULL, oracle_worker, &jobs[t]) != 0) {
            /* fall back to running this share inline; arithmetic is unchanged */
            oracle_worker(&jobs[t]);
            th[t] = 0;
            continue;
        }
        ++started;
    }
    oracle_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (th[t]) pthread_join(th[t], NULL);
    return started + 1;
}

/*
 * Full mode: C (M x N, row stride ldc, fp64) = the definition above for every
 * (m, n).  Returns the number of threads used, or -1 on bad arguments.
 */
int oracle_gemm_f64(const uint16_t *A, const uint16_t *B, double *C,
                    int64_t M, int64_t N, int64_t K,
                    int64_t lda, int64_t ldb, int64_t ldc, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < K || ldc < N) return -1;
    if (M == 0 || N == 0) return 0;
    oracle_job base;
    memset(&base, 0, sizeof base);
    base.A = A; base.B = B; base.C = C;
    base.N = N; base.K = K; base.lda = lda; base.ldb = ldb; base.ldc = ldc;
    base.rows = NULL; base.nrows = M;
    base.cols = NULL; base.ncols = N;
    return run_jobs(base, nthreads);
}

/*
 * Sampled mode: out[i][c] (nrows x ncols, dense) = the definition above at
 * (rows[i], cols[c]).  Returns the number of threads used, or -1.
 */
int oracle_gemm_sampled_f64(const uint16_t *A, const uint16_t *B, double *out,
                            const int64_t *rows, int64_t nrows,
                            const int64_t *cols, int64_t ncols,
                            int64_t K, int64_t lda, int64_t ldb, int nthreads)
{
    if (nrows < 0 || ncols < 0 || K < 0 || lda < K || ldb < K) return -1;
    if (nrows == 0 || ncols == 0) return 0;
    oracle_job base;
    memset(&base, 0, sizeof base);
    base.A = A; base.B = B; base.C = out;
    base.N = ncols; base.K = K; base.lda = lda; base.ldb = ldb; base.ldc = ncols;
    base.rows = rows; base.nrows = nrows;
    base.cols = cols; base.ncols = ncols;
    return run_jobs(base, nthreads);
}
