/*
 * gemm_oracle.c -- the plain, slow CPU oracle for dense GEMM, C = A * B.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no header, helper, table or
 * constant with the CUDA library.
 *
 * What it computes (the definition, written out):
 *   C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j]
 *     "GEMM" (inference-book, Part 4), opening section, the element formula;
 *     "GEMM Optimization" (infra.bea.ai), section 1 "The Problem".
 *   A is M x K, B is K x N, C is M x N, all row-major with leading
 *   dimensions lda, ldb, ldc (row r of A starts at A + r*lda).
 *     "How a Matrix Multiply Runs on a GPU", "Level 0: one thread per output"
 *     (row-major indexing A[row*K+k], B[k*N+col]).
 *
 * Precision: every product and every sum is taken in IEEE double, from the
 * exact input values (FP32 as given; BF16 widened exactly by placing its 16
 * bits in the top half of an FP32 word).  This is the double-precision CPU
 * reference the GPU results are checked against in "A06 -- Tiled Matrix
 * Multiply (GEMM)", section 4 "Hands-On Labs", Lab 1.
 *
 * Alongside C it can return S[i][j] = sum_k |A[i][k] * B[k][j]|, the scale
 * that the elementwise error bound |C_gpu - C| <= rtol*S + atol is taken
 * against.
 *
 * Loop order is i, k, j: for each row i the output row itself is the
 * running double accumulator, and for each k the whole row B[k][*] is added
 * in, scaled by A[i][k].  No blocking, no reordering of the sum over k: the
 * sum for every (i, j) is taken in increasing k.  Rows are independent, so
 * they are spread over OpenMP threads when the library is built with
 * -fopenmp; that changes nothing in any row's arithmetic.
 *
 * Empty cases: M == 0 or N == 0 writes nothing; K == 0 writes zeros (the
 * empty sum).
 *
 * Return value: 0 on success, -1 on an invalid argument (negative size, a
 * leading dimension shorter than its row, or a null pointer where data is
 * needed).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* BF16 -> double, exact: the 16 stored bits are the top half of an FP32. */
double oracle_bf16_to_double(uint16_t bits)
{
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

static int check_args(int64_t M, int64_t N, int64_t K, const void *A,
                      int64_t lda, const void *B, int64_t ldb,
                      const double *C, int64_t ldc)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (M == 0 || N == 0) return 0;
    if (lda < K || ldb < N || ldc < N) return -1;
    if (C == NULL) return -1;
    if (K > 0 && (A == NULL || B == NULL)) return -1;
    return 0;
}

/* The two element types differ only in how one input value is read. */
#define ORACLE_GEMM_BODY(READ_A, READ_B)                                      \
    int64_t i;                                                                \
    _Pragma("omp parallel for schedule(dynamic, 1)")                          \
    for (i = 0; i < M; ++i) {                                                 \
        double *c_row = C + i * ldc;                                          \
        double *s_row = S ? S + i * ldc : NULL;                               \
        for (int64_t j = 0; j < N; ++j) c_row[j] = 0.0;                       \
        if (s_row)                                                            \
            for (int64_t j = 0; j < N; ++j) s_row[j] = 0.0;                   \
        for (int64_t k = 0; k < K; ++k) {                                     \
            const double a_ik = READ_A(A[i * lda + k]);                       \
            for (int64_t j = 0; j < N; ++j) {                                 \
                const double p = a_ik * READ_B(B[k * ldb + j]);               \
                c_row[j] += p;                                                \
                if (s_row) s_row[j] += fabs(p);                               \
            }                                                                 \
        }                                                                     \
    }

#define READ_F32(x) ((double)(x))
#define READ_BF16(x) oracle_bf16_to_double(x)

int oracle_gemm_f32(int64_t M, int64_t N, int64_t K,
                    const float *A, int64_t lda,
                    const float *B, int64_t ldb,
                    double *C, int64_t ldc, double *S)
{
    if (check_args(M, N, K, A, lda, B, ldb, C, ldc)) return -1;
    if (M == 0 || N == 0) return 0;
    ORACLE_GEMM_BODY(READ_F32, READ_F32)
    return 0;
}

int oracle_gemm_bf16(int64_t M, int64_t N, int64_t K,
                     const uint16_t *A, int64_t lda,
                     const uint16_t *B, int64_t ldb,
                     double *C, int64_t ldc, double *S)
{
    if (check_args(M, N, K, A, lda, B, ldb, C, ldc)) return -1;
    if (M == 0 || N == 0) return 0;
    ORACLE_GEMM_BODY(READ_BF16, READ_BF16)
    return 0;
}

/*
 * The epilogue step of the register-tiled kernel's pseudocode ("How a Matrix
 * Multiply Runs on a GPU", "Level 2": the output is alpha * acc + beta * C,
 * plus a bias and an activation) applied to an exact product:
 *   out[i][j] = act(alpha * AB[i][j] + beta * C0[i][j] + bias[j])
 * in double.  AB is the oracle's product (ld_ab), C0 the prior contents of
 * C as FP32 (NULL: treated as zero, i.e. not read), bias N floats or NULL,
 * act 0 = identity, 1 = max(x, 0), 2 = GELU, x * Phi(x) with Phi the
 * standard normal distribution function, 0.5 x (1 + erf(x / sqrt(2)))
 * (the activation named among a transformer's element-wise operations in
 * "GEMM Optimization").  Returns 0, or -1 on a bad argument.
 */
int oracle_gemm_epilogue(int64_t M, int64_t N, const double *AB, int64_t ld_ab,
                         double alpha, double beta, const float *C0,
                         int64_t ld_c0, const float *bias, int act, double *out,
                         int64_t ld_out)
{
    if (M < 0 || N < 0 || act < 0 || act > 2) return -1;
    if (M == 0 || N == 0) return 0;
    if (AB == NULL || out == NULL || ld_ab < N || ld_out < N) return -1;
    if (C0 != NULL && ld_c0 < N) return -1;
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double v = alpha * AB[i * ld_ab + j];
            if (C0 != NULL) v += beta * (double)C0[i * ld_c0 + j];
            if (bias != NULL) v += (double)bias[j];
            if (act == 1 && v < 0.0) v = 0.0;
            if (act == 2) v = 0.5 * v * (1.0 + erf(v / sqrt(2.0)));
            out[i * ld_out + j] = v;
        }
    }
    return 0;
}

/* Floating-point operation count of one GEMM: one multiply and one add per
 * (i, j, k), i.e. 2*M*N*K ("A06 -- Tiled Matrix Multiply (GEMM)", section 6,
 * Pitfall 4; "How a Matrix Multiply Runs on a GPU", "The problem and the
 * roofline"). */
double oracle_gemm_flops(int64_t M, int64_t N, int64_t K)
{
    return 2.0 * (double)M * (double)N * (double)K;
}

/* Threads the oracle's row loop will use (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
