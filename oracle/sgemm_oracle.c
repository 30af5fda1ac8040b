/*
 * CPU oracle for the single-precision matrix product. TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg may load
 * this file's library. The GPU library shares no code with it.
 *
 * What it computes: the problem statement of "LeetGPU | 02_Matrix_Multiplication"
 * (sections "Problem Description" and "CUDA / Approach"). A is M x N, B is N x K and
 * C is M x K, all row-major float32, and
 *
 *     C[m][k] = sum over n = 0 .. N-1 of A[m][n] * B[n][k],
 *
 * addressed as A[m*N + n], B[n*K + k], C[m*K + k]. The same definition appears in
 * "CUDA 学习笔记 Matrix Multiplication" section "1. 题目含义".
 *
 * How: a plain triple loop. Every product is formed in double from the float inputs
 * (exact, since two 24-bit significands need at most 48 bits) and summed in double
 * with n ascending, following the double-precision CPU reference of "分块计算与矩阵乘法"
 * section "3. 完整对照程序". The loops run in m, n, k order with a per-row double
 * accumulator vector, which keeps each element's summation order (n ascending) the
 * same as the textbook m, k, n nest while reading B row by row. Rows are split across
 * threads; each element is summed by one thread in one order, so the result does not
 * depend on the thread count.
 *
 * In the same pass it forms S[m][k] = sum over n of |A[m][n]| * |B[n][k]|, the scale
 * of the elementwise error bounds |C_gpu - C| <= tol * S.
 *
 * Parity pins (tests/test_oracle.py): the pages' three worked examples, exact rational
 * sums on tiny shapes, integer inputs against exact integer products, identity,
 * permutation and transpose invariants, and closed forms.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

typedef struct {
    const float* A;
    const float* B;
    double* C;
    double* S;
    int64_t M, N, K;
    int64_t row_begin, row_end;
    int status;
} rows_job;

static void* run_rows(void* arg) {
    rows_job* job = (rows_job*)arg;
    const int64_t N = job->N, K = job->K;
    double* acc = (double*)malloc((size_t)K * sizeof(double));
    double* acc_abs = job->S ? (double*)malloc((size_t)K * sizeof(double)) : NULL;
    if (!acc || (job->S && !acc_abs)) {
        free(acc);
        free(acc_abs);
        job->status = -1;
        return NULL;
    }
    for (int64_t m = job->row_begin; m < job->row_end; ++m) {
        for (int64_t k = 0; k < K; ++k) acc[k] = 0.0;
        if (acc_abs)
            for (int64_t k = 0; k < K; ++k) acc_abs[k] = 0.0;
        const float* a_row = job->A + m * N;
        for (int64_t n = 0; n < N; ++n) {
            const double a = (double)a_row[n];
            const float* b_row = job->B + n * K;
            for (int64_t k = 0; k < K; ++k) acc[k] += a * (double)b_row[k];
            if (acc_abs) {
                const double a_abs = fabs(a);
                for (int64_t k = 0; k < K; ++k) acc_abs[k] += a_abs * fabs((double)b_row[k]);
            }
        }
        for (int64_t k = 0; k < K; ++k) job->C[m * K + k] = acc[k];
        if (acc_abs)
            for (int64_t k = 0; k < K; ++k) job->S[m * K + k] = acc_abs[k];
    }
    free(acc);
    free(acc_abs);
    job->status = 0;
    return NULL;
}

/* Full product. C (M*K doubles) is required, S (M*K doubles) may be NULL.
 * Returns 0, or -1 on bad arguments or a failed allocation. */
int oracle_gemm(const float* A, const float* B, double* C, double* S,
                int64_t M, int64_t N, int64_t K, int threads) {
    if (!A || !B || !C || M < 1 || N < 1 || K < 1) return -1;
    if (threads < 1) threads = 1;
    if (threads > M) threads = (int)M;
    pthread_t* tid = (pthread_t*)malloc((size_t)threads * sizeof(pthread_t));
    rows_job* jobs = (rows_job*)malloc((size_t)threads * sizeof(rows_job));
    char* spawned = (char*)calloc((size_t)threads, 1);
    if (!tid || !jobs || !spawned) {
        free(tid);
        free(jobs);
        free(spawned);
        return -1;
    }
    for (int t = 0; t < threads; ++t) {
        jobs[t] = (rows_job){A, B, C, S, M, N, K, M * t / threads, M * (t + 1) / threads, -1};
        /* the last slice, and any slice whose thread could not be started, runs here */
        if (t < threads - 1 && pthread_create(&tid[t], NULL, run_rows, &jobs[t]) == 0)
            spawned[t] = 1;
        else
            run_rows(&jobs[t]);
    }
    int rc = 0;
    for (int t = 0; t < threads; ++t) {
        if (spawned[t]) pthread_join(tid[t], NULL);
        if (jobs[t].status != 0) rc = -1;
    }
    free(tid);
    free(jobs);
    free(spawned);
    return rc;
}

/* Selected entries, each summed on its own: out_C[i] = C[rows[i]][cols[i]] and
 * out_S[i] = S[rows[i]][cols[i]] (out_S may be NULL). Same order of summation as
 * oracle_gemm, so the two agree bit for bit. Returns 0 or -1. */
int oracle_entries(const float* A, const float* B, int64_t M, int64_t N, int64_t K,
                   const int64_t* rows, const int64_t* cols, int64_t count,
                   double* out_C, double* out_S) {
    if (!A || !B || !rows || !cols || !out_C || M < 1 || N < 1 || K < 1 || count < 0)
        return -1;
    for (int64_t i = 0; i < count; ++i) {
        const int64_t m = rows[i], k = cols[i];
        if (m < 0 || m >= M || k < 0 || k >= K) return -1;
        double c = 0.0, s = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            const double a = (double)A[m * N + n];
            const double b = (double)B[n * K + k];
            c += a * b;
            s += fabs(a) * fabs(b);
        }
        out_C[i] = c;
        if (out_S) out_S[i] = s;
    }
    return 0;
}
