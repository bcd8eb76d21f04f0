/*
 * CPU oracle for single-precision GEMM.  TEST INFRASTRUCTURE ONLY: the tests,
 * the smoke check and the CPU-baseline leg of the benchmark call it; the
 * product library never links, loads or calls it, and it shares no code,
 * header or constant with the CUDA path.
 *
 * What it computes is the plain definition of GEMM
 * ("CUDA GEMM operator performance optimization", section 1.1; DD2360
 * workbook, section 9.4 "Matrix multiply"):
 *
 *     C[i][j] = sum_{k=0}^{K-1} opA[i][k] * opB[k][j]
 *
 * with the sum taken in fp64 in ascending k and rounded once to fp32 (a C
 * cast, round-to-nearest-even).  This is the "CPU reference with double
 * accumulation" of the DD2360 workbook, section 14.3 lab.  Every product of
 * two floats is exact in fp64 (24 + 24 significant bits <= 53), so the only
 * roundings are those of the fp64 running sum and the final cast; whether the
 * compiler fuses the multiply into the add cannot change any result.
 *
 * The loops run i -> k -> j with one fp64 accumulator per output of the row.
 * Each accumulator still receives its K terms in ascending k, i.e. exactly
 * the arithmetic of the i -> j -> k triple loop; only the loop nest order
 * differs, which lets the inner loop stream a row of B.
 *
 * Alongside C it can produce the tolerance scale S[i][j] = sum_k |a_ik||b_kj|
 * (fp64, same order), used by the elementwise acceptance bound
 * |C - C_ref| <= 1e-5 * S + 1e-6.
 *
 * Layout (row-major): opA(i,k) = A[i*lda+k] (transA=0) or A[k*lda+i]
 * (transA=1); opB(k,j) = B[k*ldb+j] (transB=0) or B[j*ldb+k] (transB=1);
 * C(i,j) = C[i*ldc+j].  Padding columns of A, B and C are never touched.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t M, N, K;
    const float *A; int64_t lda; int transA;
    const float *B; int64_t ldb; int transB;
    float *C; int64_t ldc;
    double *S; int64_t lds;
    int64_t row_begin, row_end;
    int status;
} oracle_job;

static double op_a(const oracle_job *j, int64_t i, int64_t k) {
    return j->transA ? (double)j->A[k * j->lda + i] : (double)j->A[i * j->lda + k];
}

static double op_b(const oracle_job *j, int64_t k, int64_t c) {
    return j->transB ? (double)j->B[c * j->ldb + k] : (double)j->B[k * j->ldb + c];
}

static void *oracle_rows(void *arg) {
    oracle_job *j = (oracle_job *)arg;
    const int64_t N = j->N;
    double *acc = (double *)calloc((size_t)(N > 0 ? N : 1), sizeof(double));
    double *sab = j->S ? (double *)calloc((size_t)(N > 0 ? N : 1), sizeof(double)) : NULL;
    if (!acc || (j->S && !sab)) {
        free(acc);
        free(sab);
        j->status = 1;
        return NULL;
    }
    for (int64_t i = j->row_begin; i < j->row_end; ++i) {
        for (int64_t c = 0; c < N; ++c) acc[c] = 0.0;
        if (sab) for (int64_t c = 0; c < N; ++c) sab[c] = 0.0;
        for (int64_t k = 0; k < j->K; ++k) {
            const double a = op_a(j, i, k);
            for (int64_t c = 0; c < N; ++c) acc[c] += a * op_b(j, k, c);
            if (sab) {
                const double aa = fabs(a);
                for (int64_t c = 0; c < N; ++c) sab[c] += aa * fabs(op_b(j, k, c));
            }
        }
        for (int64_t c = 0; c < N; ++c) j->C[i * j->ldc + c] = (float)acc[c];
        if (sab) for (int64_t c = 0; c < N; ++c) j->S[i * j->lds + c] = sab[c];
    }
    free(acc);
    free(sab);
    j->status = 0;
    return NULL;
}

/* Full product.  S (nullable) receives sum_k |a||b| with row stride lds.
 * nthreads <= 0 means one thread.  Returns 0 on success, 1 on allocation or
 * thread failure, 2 on bad arguments. */
int oracle_sgemm(int64_t M, int64_t N, int64_t K,
                 const float *A, int64_t lda, int transA,
                 const float *B, int64_t ldb, int transB,
                 float *C, int64_t ldc, double *S, int64_t lds, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || (transA != 0 && transA != 1) || (transB != 0 && transB != 1))
        return 2;
    if (M == 0 || N == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > M) nthreads = (int)M;
    if (nthreads > 256) nthreads = 256;
    oracle_job jobs[256];
    pthread_t tids[256];
    int started[256];
    for (int t = 0; t < nthreads; ++t) {
        oracle_job *j = &jobs[t];
        j->M = M; j->N = N; j->K = K;
        j->A = A; j->lda = lda; j->transA = transA;
        j->B = B; j->ldb = ldb; j->transB = transB;
        j->C = C; j->ldc = ldc; j->S = S; j->lds = lds;
        j->row_begin = M * t / nthreads;
        j->row_end = M * (t + 1) / nthreads;
        j->status = 1;
        started[t] = 0;
    }
    for (int t = 1; t < nthreads; ++t)
        started[t] = pthread_create(&tids[t], NULL, oracle_rows, &jobs[t]) == 0;
    oracle_rows(&jobs[0]);
    int status = jobs[0].status;
    for (int t = 1; t < nthreads; ++t) {
        if (started[t]) {
            pthread_join(tids[t], NULL);
            status |= jobs[t].status;
        } else {
            oracle_rows(&jobs[t]);
            status |= jobs[t].status;
        }
    }
    return status;
}

/* Strided batch: problem z uses A + z*strideA, B + z*strideB, C + z*strideC
 * (and S + z*strideS).  Each problem is the full product above. */
int oracle_sgemm_strided_batched(int64_t M, int64_t N, int64_t K,
                                 const float *A, int64_t lda, int64_t strideA, int transA,
                                 const float *B, int64_t ldb, int64_t strideB, int transB,
                                 float *C, int64_t ldc, int64_t strideC,
                                 double *S, int64_t lds, int64_t strideS,
                                 int64_t batch, int nthreads) {
    if (batch < 0) return 2;
    for (int64_t z = 0; z < batch; ++z) {
        int st = oracle_sgemm(M, N, K, A + z * strideA, lda, transA, B + z * strideB, ldb, transB,
                              C + z * strideC, ldc, S ? S + z * strideS : NULL, lds, nthreads);
        if (st) return st;
    }
    return 0;
}

/* Selected outputs, one dot product each: out[t] = C(rows[t], cols[t]) and
 * sabs[t] (nullable) its tolerance scale.  Lets full-size problems be checked
 * on a sample of outputs. */
int oracle_sgemm_entries(int64_t M, int64_t N, int64_t K,
                         const float *A, int64_t lda, int transA,
                         const float *B, int64_t ldb, int transB,
                         int64_t count, const int64_t *rows, const int64_t *cols,
                         float *out, double *sabs) {
    if (M < 0 || N < 0 || K < 0 || count < 0) return 2;
    oracle_job j;
    memset(&j, 0, sizeof j);
    j.M = M; j.N = N; j.K = K;
    j.A = A; j.lda = lda; j.transA = transA;
    j.B = B; j.ldb = ldb; j.transB = transB;
    for (int64_t t = 0; t < count; ++t) {
        const int64_t i = rows[t], c = cols[t];
        if (i < 0 || i >= M || c < 0 || c >= N) return 2;
        double acc = 0.0, s = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = op_a(&j, i, k), b = op_b(&j, k, c);
            acc += a * b;
            s += fabs(a) * fabs(b);
        }
        out[t] = (float)acc;
        if (sabs) sabs[t] = s;
    }
    return 0;
}

/* The general form: C_out = alpha * op(A) op(B) + beta * C_in + bias (bias
 * broadcast along rows, one value per output column).  Everything is formed
 * in fp64 (the product sum in ascending k as above) and rounded once to fp32.
 * beta == 0 means C_in is not read (it may hold anything); bias may be NULL.
 * S (nullable) receives the tolerance scale
 * |alpha| * sum_k |a||b| + |beta| * |C_in| + |bias|.
 * This is the fully connected layer Y = XW + b that "CUDA GEMM operator
 * performance optimization" section 1.2 names, with the BLAS-style scaling. */
int oracle_sgemm_ex(int64_t M, int64_t N, int64_t K, double alpha,
                    const float *A, int64_t lda, int transA,
                    const float *B, int64_t ldb, int transB,
                    double beta, const float *C_in, int64_t ldc_in,
                    const float *bias, float *C_out, int64_t ldc_out,
                    double *S, int64_t lds) {
    if (M < 0 || N < 0 || K < 0) return 2;
    if (M == 0 || N == 0) return 0;
    /* one dot product per output, in ascending k, kept in fp64 until the end */
    oracle_job j;
    memset(&j, 0, sizeof j);
    j.M = M; j.N = N; j.K = K;
    j.A = A; j.lda = lda; j.transA = transA;
    j.B = B; j.ldb = ldb; j.transB = transB;
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t c = 0; c < N; ++c) {
            double acc = 0.0, s = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double a = op_a(&j, i, k), b = op_b(&j, k, c);
                acc += a * b;
                s += fabs(a) * fabs(b);
            }
            double v = alpha * acc;
            double scale = fabs(alpha) * s;
            if (beta != 0.0) {
                const double cin = (double)C_in[i * ldc_in + c];
                v += beta * cin;
                scale += fabs(beta) * fabs(cin);
            }
            if (bias) {
                v += (double)bias[c];
                scale += fabs((double)bias[c]);
            }
            C_out[i * ldc_out + c] = (float)v;
            if (S) S[i * lds + c] = scale;
        }
    }
    return 0;
}
