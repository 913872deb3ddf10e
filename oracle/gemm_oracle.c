/*
 * Plain CPU oracle for the dense product C = A·B (test infrastructure only).
 *
 * This file is the checker that the CUDA path is compared against. It is not
 * part of the product: only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg load it. It shares no code, header, table or
 * constant with the CUDA sources.
 *
 * What it computes, and where that is defined:
 *   - "4.1 CUDA GEMM 算子性能优化", §1.1 (GEMM 的定义): C = A × B with A of
 *     shape M×K, B of shape K×N, C of shape M×N, i.e.
 *         C[i][j] = sum over k of A[i][k] · B[k][j].
 *   - same page, §3.1 (朴素实现): one output element is the inner product of
 *     row i of A and column j of B, walked along k from 0 to K-1, with A and
 *     B row-major (A[i*lda + k], B[k*ldb + j]).
 *   - "流水化 GPU 内核", step 5 (验证正确性): pipelining only reorders the
 *     loads, it does not change the arithmetic, so the correct result of the
 *     pipelined kernel is this plain definition.
 *
 * Arithmetic: every input is first decoded to the exact value that the
 * tensor cores consume (bf16 exactly; fp32 reduced to TF32; int8 exactly),
 * then the triple loop accumulates in IEEE fp64 (int64 for int8), rows in
 * i-k-j order so that row i of C is a running sum over k = 0, 1, ..., K-1.
 * Alongside C it can return S[i][j] = sum over k of |A[i][k]·B[k][j]|,
 * the scale against which floating-point tolerances are stated.
 *
 * Every product of two decoded bf16 (8-bit significand) or TF32 (11-bit
 * significand) values is exact in fp64, so the only rounding in C is the fp64
 * summation itself. Rows are independent, so they are spread over OpenMP
 * threads; each row is still summed serially in k order.
 *
 * Compiled with -ffp-contract=off so that the same source gives the same bits
 * on x86-64 and aarch64 hosts.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- input decoding ---------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32: widen by 16 zero bits. */
static double dec_bf16(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* TF32 keeps the sign, the 8 exponent bits and the top 10 of the 23 stored
 * mantissa bits of a binary32.
 *   mode 0: truncate (the low 13 bits are ignored);
 *   mode 1: round to nearest, ties to even, at that position (NaN/Inf kept).
 */
static double dec_tf32(float x, int mode) {
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if (mode == 0) {
        u &= 0xFFFFE000u;
    } else if ((u & 0x7F800000u) != 0x7F800000u) {
        uint32_t keep_lsb = (u >> 13) & 1u;
        u += 0x00000FFFu + keep_lsb;
        u &= 0xFFFFE000u;
    }
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

void oracle_decode_bf16(const uint16_t* in, double* out, long n) {
    for (long i = 0; i < n; ++i) out[i] = dec_bf16(in[i]);
}

void oracle_decode_tf32(const float* in, double* out, long n, int mode) {
    for (long i = 0; i < n; ++i) out[i] = dec_tf32(in[i], mode);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the following calls (n >= 1); used to time the oracle on one core. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---- the definition, in fp64 -------------------------------------------
 * Rows [i0, i1) and columns [j0, j1) of C = A·B, where A is given by a row
 * decoder and B already decoded to doubles (Bd, K rows, ldbd columns, holding
 * columns j0..j1-1 of B). C and S are written row-major with strides ldc/lds
 * and hold (i1-i0) rows of (j1-j0) columns. S may be NULL.
 */
typedef double (*row_getter)(const void* A, long lda, long i, long k, int mode);

static double get_bf16(const void* A, long lda, long i, long k, int mode) {
    (void)mode;
    return dec_bf16(((const uint16_t*)A)[i * lda + k]);
}

static double get_tf32(const void* A, long lda, long i, long k, int mode) {
    return dec_tf32(((const float*)A)[i * lda + k], mode);
}

static void gemm_f64_rows(long K, const void* A, long lda, row_getter getA, int mode,
                          const double* Bd, long ldbd, long i0, long i1, long ncols,
                          double* C, long ldc, double* S, long lds) {
    long i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = i0; i < i1; ++i) {
        double* c = C + (i - i0) * ldc;
        double* s = S ? S + (i - i0) * lds : NULL;
        for (long j = 0; j < ncols; ++j) c[j] = 0.0;
        if (s)
            for (long j = 0; j < ncols; ++j) s[j] = 0.0;
        for (long k = 0; k < K; ++k) {
            const double a = getA(A, lda, i, k, mode);
            const double* b = Bd + k * ldbd;
            for (long j = 0; j < ncols; ++j) c[j] += a * b[j];
            if (s)
                for (long j = 0; j < ncols; ++j) s[j] += fabs(a * b[j]);
        }
    }
}

static int check_args(long M, long N, long K, const void* A, long lda, const void* B, long ldb,
                      long i0, long i1, long j0, long j1, const void* C, long ldc) {
    if (M < 0 || N < 0 || K < 0) return 2;
    if (!A || !B || !C) return 1;
    if (lda < K || ldb < N) return 3;
    if (i0 < 0 || i1 > M || i0 > i1 || j0 < 0 || j1 > N || j0 > j1) return 2;
    if (ldc < j1 - j0) return 3;
    return 0;
}

/* bf16 inputs given as their 16-bit patterns; fp64 result. */
int oracle_gemm_bf16(long M, long N, long K, const uint16_t* A, long lda, const uint16_t* B,
                     long ldb, long i0, long i1, long j0, long j1, double* C, long ldc,
                     double* S, long lds) {
    int st = check_args(M, N, K, A, lda, B, ldb, i0, i1, j0, j1, C, ldc);
    if (st) return st;
    long ncols = j1 - j0;
    double* Bd = (double*)malloc(sizeof(double) * (size_t)(K * ncols + 1));
    if (!Bd) return 9;
    for (long k = 0; k < K; ++k)
        for (long j = 0; j < ncols; ++j) Bd[k * ncols + j] = dec_bf16(B[k * ldb + j0 + j]);
    gemm_f64_rows(K, A, lda, get_bf16, 0, Bd, ncols, i0, i1, ncols, C, ldc, S, lds);
    free(Bd);
    return 0;
}

/* fp32 inputs consumed as TF32 (mode 0 truncate, 1 round-nearest-even). */
int oracle_gemm_tf32(long M, long N, long K, const float* A, long lda, const float* B, long ldb,
                     long i0, long i1, long j0, long j1, double* C, long ldc, double* S,
                     long lds, int mode) {
    int st = check_args(M, N, K, A, lda, B, ldb, i0, i1, j0, j1, C, ldc);
    if (st) return st;
    long ncols = j1 - j0;
    double* Bd = (double*)malloc(sizeof(double) * (size_t)(K * ncols + 1));
    if (!Bd) return 9;
    for (long k = 0; k < K; ++k)
        for (long j = 0; j < ncols; ++j) Bd[k * ncols + j] = dec_tf32(B[k * ldb + j0 + j], mode);
    gemm_f64_rows(K, A, lda, get_tf32, mode, Bd, ncols, i0, i1, ncols, C, ldc, S, lds);
    free(Bd);
    return 0;
}

/* Plain fp64 inputs (used to check the summation itself on exact data). */
static double get_f64(const void* A, long lda, long i, long k, int mode) {
    (void)mode;
    return ((const double*)A)[i * lda + k];
}

int oracle_gemm_f64(long M, long N, long K, const double* A, long lda, const double* B, long ldb,
                    long i0, long i1, long j0, long j1, double* C, long ldc, double* S, long lds) {
    int st = check_args(M, N, K, A, lda, B, ldb, i0, i1, j0, j1, C, ldc);
    if (st) return st;
    long ncols = j1 - j0;
    double* Bd = (double*)malloc(sizeof(double) * (size_t)(K * ncols + 1));
    if (!Bd) return 9;
    for (long k = 0; k < K; ++k)
        for (long j = 0; j < ncols; ++j) Bd[k * ncols + j] = B[k * ldb + j0 + j];
    gemm_f64_rows(K, A, lda, get_f64, 0, Bd, ncols, i0, i1, ncols, C, ldc, S, lds);
    free(Bd);
    return 0;
}

/* int8 inputs, exact int64 accumulation. */
int oracle_gemm_s8(long M, long N, long K, const int8_t* A, long lda, const int8_t* B, long ldb,
                   long i0, long i1, long j0, long j1, int64_t* C, long ldc) {
    int st = check_args(M, N, K, A, lda, B, ldb, i0, i1, j0, j1, C, ldc);
    if (st) return st;
    long ncols = j1 - j0;
    long i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = i0; i < i1; ++i) {
        int64_t* c = C + (i - i0) * ldc;
        for (long j = 0; j < ncols; ++j) c[j] = 0;
        for (long k = 0; k < K; ++k) {
            const int64_t a = (int64_t)A[i * lda + k];
            const int8_t* b = B + k * ldb + j0;
            for (long j = 0; j < ncols; ++j) c[j] += a * (int64_t)b[j];
        }
    }
    return 0;
}
