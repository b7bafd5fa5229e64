/*
 * CPU oracle for C = alpha * op(A) * op(B) + beta * C  (TEST INFRASTRUCTURE ONLY).
 *
 * This file is the correctness anchor for the GPU library, not part of it.  Only the
 * test-suite, the smoke check and the CPU-baseline leg of the benchmark may load it.  It
 * shares no code, header or table with the CUDA sources.
 *
 * What it computes (copecc.github.io "GEMM" page, section "核心问题与运算特征": the GEMM
 * form alpha*op(A)op(B)+beta*C, with A of M x K, B of K x N, C of M x N, and each C[i][j]
 * a dot product of row i of op(A) with column j of op(B); yekq.top "LeetGPU 第二题",
 * section "题目描述": C[row][col] = sum_i A[row][i] * B[i][col]):
 *
 *     S[i][j]    = sum_{k=0}^{K-1} opA(i,k) * opB(k,j)      (fp64, k in increasing order)
 *     Cout[i][j] = (float)(alpha * S[i][j] + beta * Cin[i][j])
 *
 * Storage is row-major with explicit leading dimensions (copecc "GEMM" page, section
 * "Leading Dimension (lda, ldb, ldc)": ld is the element distance between the starts of
 * consecutive rows, which may exceed the logical column count because of padding):
 *     opA(i,k) = A[i*lda + k]  (opA = N, A stored M x K)    or  A[k*lda + i]  (opA = T)
 *     opB(k,j) = B[k*ldb + j]  (opB = N, B stored K x N)    or  B[j*ldb + k]  (opB = T)
 *
 * Precision: every fp32, fp16 and bf16 input is converted to fp64 exactly, so each product
 * of two inputs is exact in fp64 (at most 24 + 24 significant bits).  Sums are taken in fp64 in k
 * order.  beta == 0 means Cin is not read at all (BLAS convention), so NaN or Inf in Cin does
 * not reach the result.  The fp16 inputs are decoded from their bit patterns by the decoder
 * below, written from the IEEE 754 binary16 definition (1 sign bit, 5 exponent bits with bias
 * 15, 10 fraction bits; exponent 0 = zero/subnormal, exponent 31 = Inf/NaN); bf16 inputs
 * (mixed precision with BF16 inputs, copecc "GEMM" page, section "Batched 执行与混合精度") are
 * the upper 16 bits of an IEEE binary32 pattern.
 *
 * Optionally the oracle also returns absdot[i][j] = sum_k |opA(i,k) * opB(k,j)|, the
 * quantity the acceptance bound of the parity tests is written in.
 *
 * Rows are split over POSIX threads; each output element is still one sequential k loop,
 * so the thread count never changes a result.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OP_N 0
#define ORACLE_OP_T 1

/* IEEE 754 binary16 -> double, exact. */
double gemm_oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24); /* subnormal: frac * 2^-10 * 2^-14 */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(frac | 0x400), expo - 25); /* (1 + frac/1024) * 2^(expo-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 -> double, exact: the 16 bits are the upper half of an IEEE binary32 pattern
 * (1 sign bit, 8 exponent bits with bias 127, 7 fraction bits). */
double gemm_oracle_bf16_to_double(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

typedef struct {
    int dtype; /* 0 = fp32 inputs, 1 = fp16 inputs, 2 = bf16 inputs */
    int opA, opB;
    int64_t M, N, K;
    double alpha, beta;
    const void *A;
    int64_t lda;
    const void *B;
    int64_t ldb;
    const float *Cin;
    int64_t ldcin;
    float *Cout;
    int64_t ldc;
    double *absdot;
    int64_t ldabs;
    /* point mode: only the listed (row, col) pairs are computed */
    const int64_t *rows, *cols;
    int64_t npts;
    float *pts_out;
    double *pts_abs;
    int64_t begin, end; /* row range (full mode) or point range (point mode) */
    int err;            /* set by a worker that could not get its scratch row */
} job_t;

static inline double load_in(const job_t *j, const void *base, int64_t idx)
{
    if (j->dtype == 0) return (double)((const float *)base)[idx];
    if (j->dtype == 2) return gemm_oracle_bf16_to_double(((const uint16_t *)base)[idx]);
    return gemm_oracle_half_to_double(((const uint16_t *)base)[idx]);
}

static inline double opA_at(const job_t *j, int64_t i, int64_t k)
{
    return load_in(j, j->A, j->opA == ORACLE_OP_N ? i * j->lda + k : k * j->lda + i);
}

static inline double opB_at(const job_t *j, int64_t k, int64_t c)
{
    return load_in(j, j->B, j->opB == ORACLE_OP_N ? k * j->ldb + c : c * j->ldb + k);
}

/* One element: the dot product in k order, then the alpha/beta update. */
static void element(const job_t *j, int64_t i, int64_t c, float *out, double *abs_out)
{
    double s = 0.0, sa = 0.0;
    for (int64_t k = 0; k < j->K; ++k) {
        double p = opA_at(j, i, k) * opB_at(j, k, c);
        s += p;
        sa += fabs(p);
    }
    double r = j->alpha * s;
    if (j->beta != 0.0) r += j->beta * (double)j->Cin[i * j->ldcin + c];
    *out = (float)r;
    if (abs_out) *abs_out = sa;
}

/* Full mode for op(B) = N: i-k-j order with an fp64 row accumulator.  For each (i, j) the
 * terms are still added in increasing k, exactly as in element(). */
static void rows_opBN(const job_t *j, double *acc, double *aacc)
{
    for (int64_t i = j->begin; i < j->end; ++i) {
        for (int64_t c = 0; c < j->N; ++c) { acc[c] = 0.0; aacc[c] = 0.0; }
        for (int64_t k = 0; k < j->K; ++k) {
            double a = opA_at(j, i, k);
            if (j->dtype == 0) {
                const float *brow = (const float *)j->B + k * j->ldb;
                if (j->absdot) {
                    for (int64_t c = 0; c < j->N; ++c) {
                        double p = a * (double)brow[c];
                        acc[c] += p;
                        aacc[c] += fabs(p);
                    }
                } else {
                    for (int64_t c = 0; c < j->N; ++c) acc[c] += a * (double)brow[c];
                }
            } else {
                const uint16_t *brow = (const uint16_t *)j->B + k * j->ldb;
                for (int64_t c = 0; c < j->N; ++c) {
                    double p = a * (j->dtype == 2 ? gemm_oracle_bf16_to_double(brow[c])
                                                  : gemm_oracle_half_to_double(brow[c]));
                    acc[c] += p;
                    aacc[c] += fabs(p);
                }
            }
        }
        for (int64_t c = 0; c < j->N; ++c) {
            double r = j->alpha * acc[c];
            if (j->beta != 0.0) r += j->beta * (double)j->Cin[i * j->ldcin + c];
            j->Cout[i * j->ldc + c] = (float)r;
            if (j->absdot) j->absdot[i * j->ldabs + c] = aacc[c];
        }
    }
}

static void *worker(void *arg)
{
    job_t *j = (job_t *)arg;
    if (j->rows) {
        for (int64_t p = j->begin; p < j->end; ++p)
            element(j, j->rows[p], j->cols[p], &j->pts_out[p], j->pts_abs ? &j->pts_abs[p] : NULL);
        return NULL;
    }
    if (j->opB == ORACLE_OP_N) {
        double *acc = (double *)malloc(sizeof(double) * (size_t)(j->N > 0 ? j->N : 1));
        double *aacc = (double *)malloc(sizeof(double) * (size_t)(j->N > 0 ? j->N : 1));
        if (acc && aacc) rows_opBN(j, acc, aacc);
        else j->err = 1;
        free(acc);
        free(aacc);
        return NULL;
    }
    for (int64_t i = j->begin; i < j->end; ++i)
        for (int64_t c = 0; c < j->N; ++c)
            element(j, i, c, &j->Cout[i * j->ldc + c],
                    j->absdot ? &j->absdot[i * j->ldabs + c] : NULL);
    return NULL;
}

static int run(job_t *tmpl, int64_t units, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    if (units < nthreads) nthreads = (int)(units > 0 ? units : 1);
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return 1; }
    char *joined = (char *)calloc((size_t)nthreads, 1);
    if (!joined) { free(jobs); free(th); return 1; }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *tmpl;
        jobs[t].begin = units * t / nthreads;
        jobs[t].end = units * (t + 1) / nthreads;
        /* a thread that cannot be started runs its share inline */
        if (nthreads == 1 || pthread_create(&th[t], NULL, worker, &jobs[t]) != 0) worker(&jobs[t]);
        else joined[t] = 1;
    }
    int err = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (joined[t]) pthread_join(th[t], NULL);
        err |= jobs[t].err;
    }
    free(joined);
    free(jobs);
    free(th);
    return err;
}

static int check_args(int opA, int opB, int64_t M, int64_t N, int64_t K, int64_t lda,
                      int64_t ldb)
{
    if (M < 0 || N < 0 || K < 0) return 1;
    if ((opA != ORACLE_OP_N && opA != ORACLE_OP_T) || (opB != ORACLE_OP_N && opB != ORACLE_OP_T)) return 1;
    if (lda < (opA == ORACLE_OP_N ? K : M) || ldb < (opB == ORACLE_OP_N ? N : K)) return 1;
    return 0;
}

static int full(int dtype, int opA, int opB, int64_t M, int64_t N, int64_t K, double alpha,
                const void *A, int64_t lda, const void *B, int64_t ldb, double beta,
                const float *Cin, int64_t ldcin, float *Cout, int64_t ldc, double *absdot,
                int64_t ldabs, int nthreads)
{
    if (check_args(opA, opB, M, N, K, lda, ldb) || ldc < N) return 1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.dtype = dtype; j.opA = opA; j.opB = opB; j.M = M; j.N = N; j.K = K;
    j.alpha = alpha; j.beta = beta; j.A = A; j.lda = lda; j.B = B; j.ldb = ldb;
    j.Cin = Cin; j.ldcin = ldcin; j.Cout = Cout; j.ldc = ldc; j.absdot = absdot; j.ldabs = ldabs;
    return run(&j, M, nthreads);
}

static int points(int dtype, int opA, int opB, int64_t M, int64_t N, int64_t K, double alpha,
                  const void *A, int64_t lda, const void *B, int64_t ldb, double beta,
                  const float *Cin, int64_t ldcin, const int64_t *rows, const int64_t *cols,
                  int64_t npts, float *out, double *abs_out, int nthreads)
{
    if (check_args(opA, opB, M, N, K, lda, ldb)) return 1;
    for (int64_t p = 0; p < npts; ++p)
        if (rows[p] < 0 || rows[p] >= M || cols[p] < 0 || cols[p] >= N) return 1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.dtype = dtype; j.opA = opA; j.opB = opB; j.M = M; j.N = N; j.K = K;
    j.alpha = alpha; j.beta = beta; j.A = A; j.lda = lda; j.B = B; j.ldb = ldb;
    j.Cin = Cin; j.ldcin = ldcin; j.rows = rows; j.cols = cols; j.npts = npts;
    j.pts_out = out; j.pts_abs = abs_out;
    return run(&j, npts, nthreads);
}

int gemm_oracle_f32(int opA, int opB, int64_t M, int64_t N, int64_t K, double alpha,
                    const float *A, int64_t lda, const float *B, int64_t ldb, double beta,
                    const float *Cin, int64_t ldcin, float *Cout, int64_t ldc, double *absdot,
                    int64_t ldabs, int nthreads)
{
    return full(0, opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, Cin, ldcin, Cout, ldc,
                absdot, ldabs, nthreads);
}

int gemm_oracle_f16(int opA, int opB, int64_t M, int64_t N, int64_t K, double alpha,
                    const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb, double beta,
                    const float *Cin, int64_t ldcin, float *Cout, int64_t ldc, double *absdot,
                    int64_t ldabs, int nthreads)
{
    return full(1, opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, Cin, ldcin, Cout, ldc,
                absdot, ldabs, nthreads);
}

int gemm_oracle_bf16(int opA, int opB, int64_t M, int64_t N, int64_t K, double alpha,
                     const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb, double beta,
                     const float *Cin, int64_t ldcin, float *Cout, int64_t ldc, double *absdot,
                     int64_t ldabs, int nthreads)
{
    return full(2, opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, Cin, ldcin, Cout, ldc,
                absdot, ldabs, nthreads);
}

int gemm_oracle_bf16_points(int opA, int opB, int64_t M, int64_t N, int64_t K, double alpha,
                            const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                            double beta, const float *Cin, int64_t ldcin, const int64_t *rows,
                            const int64_t *cols, int64_t npts, float *out, double *abs_out,
                            int nthreads)
{
    return points(2, opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, Cin, ldcin, rows, cols,
                  npts, out, abs_out, nthreads);
}

int gemm_oracle_f32_points(int opA, int opB, int64_t M, int64_t N, int64_t K, double alpha,
                           const float *A, int64_t lda, const float *B, int64_t ldb,
                           double beta, const float *Cin, int64_t ldcin, const int64_t *rows,
                           const int64_t *cols, int64_t npts, float *out, double *abs_out,
                           int nthreads)
{
    return points(0, opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, Cin, ldcin, rows, cols,
                  npts, out, abs_out, nthreads);
}

int gemm_oracle_f16_points(int opA, int opB, int64_t M, int64_t N, int64_t K, double alpha,
                           const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                           double beta, const float *Cin, int64_t ldcin, const int64_t *rows,
                           const int64_t *cols, int64_t npts, float *out, double *abs_out,
                           int nthreads)
{
    return points(1, opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, Cin, ldcin, rows, cols,
                  npts, out, abs_out, nthreads);
}
