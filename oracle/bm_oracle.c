/*
 * CPU oracle for the BF16 BLAS3 hot path: GEMM and SYRK, plain triple loops
 * accumulating in double.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls
 * this file; only the tests, the smoke check and the bench's CPU-baseline leg
 * do. It shares no code with the CUDA library.
 *
 * What is computed (the BLAS3 statement of the local compute in "BLASMp
 * development notes", section 1, and the GEMM that the "cp.async / ldmatrix
 * ablation plan", section 2, dissects):
 *
 *   GEMM:  C[i][j] = alpha * sum_p op(A)[i][p] * op(B)[p][j] + beta * C[i][j]
 *          op(A) is m x k, op(B) is k x n, all matrices row-major.
 *   SYRK:  C[i][j] = alpha * sum_p op(A)[i][p] * op(A)[j][p] + beta * C[i][j]
 *          for (i, j) in one triangle of the n x n matrix C; op(A) is n x k
 *          ("SYRK main compute done with a GEMM", BLASMp notes, stage B).
 *   SYR2K: C[i][j] = alpha * (sum_p op(A)[i][p] * op(B)[j][p]
 *                             + sum_p op(B)[i][p] * op(A)[j][p]) + beta * C[i][j]
 *          on one triangle; op(A), op(B) are n x k (the SYR2K operator of
 *          BLASMp notes, stage D; the BLAS rank-2k update).
 *
 *   GEMM, FP8 E4M3 operands: C[i][j] = alpha * sum_p A[i][p] * B[j][p] + beta * C[i][j]
 *          with A [m, k] and B [n, k] holding E4M3 codes (the all-E4M3 inputs,
 *          FP32-accumulated products of the FP8 paths in "fused A2A/GEMM
 *          Perfetto profile protocol", FP8 section).
 *
 *   GEMM, MXFP8 operands (the SM103 MXFP8 GEMM of the same page: E4M3 data with
 *          one UE8M0 scale per group of 32 consecutive elements along K, "K32
 *          quantization group", "E32"):
 *          C[i][j] = alpha * sum_p (A[i][p] * 2^(SA[i][p/32] - 127))
 *                                * (B[j][p] * 2^(SB[j][p/32] - 127)) + beta * C[i][j]
 *          SA is [m, ceil(k/32)] and SB [n, ceil(k/32)], row-major UE8M0 codes.
 *
 *   MXFP8 quantization of a BF16 matrix X [rows, k] (the page's "W quantize
 *          BF16 -> MXFP8" step: per group of 32 along K, amax reduction, UE8M0
 *          scale, E4M3 conversion). The page names the steps, not the rule; the
 *          rule here is the OCP Microscaling (MX) v1.0 conversion: shared
 *          exponent e = floor(log2(amax)) - 8 (8 = the largest E4M3 exponent),
 *          clamped to [-127, 127], scale code e + 127, element = X / 2^e rounded
 *          to the nearest E4M3 value, ties to even, magnitudes above 448
 *          saturated to 448. A group of zeros gets code 0; a group holding a
 *          NaN or an infinity gets code 255 (NaN) and NaN elements (0x7F).
 *
 * Alongside each value the oracle returns bound[i][j] = sum_p |product|, the
 * scale against which the tolerance max|C - C_ref| <= 1e-3 * |alpha| * bound
 * is stated.
 *
 * BLAS conventions (the plainest reading of "BLAS3"): when alpha == 0 or
 * k == 0 the products are not formed and A is not read; when beta == 0 the
 * input C is not read. Storage: element (r, c) of a row-major matrix X with
 * leading dimension ld sits at X[r * ld + c]. op(X) = X for trans == 0 and
 * X^T for trans == 1.
 *
 * Products of two bf16 values are exact in double (8 + 8 significant bits),
 * and the sum runs over p in ascending order; no blocking or reordering.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> double, exact (bf16 is the top half of a float32). */
static double bf16_value(uint16_t bits)
{
    uint32_t word = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

/* FP8 E4M3 code -> double, exact: 1 sign bit, 4 exponent bits (bias 7), 3
 * mantissa bits; exponent field 0 is subnormal (m / 8 * 2^-6); S.1111.111 is NaN;
 * there are no infinities. */
static double e4m3_value(uint8_t code)
{
    int e = (code >> 3) & 0xF, m = code & 7;
    double mag;
    if (e == 0xF && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return (code & 0x80) ? -mag : mag;
}

/* UE8M0 scale code -> 2^(code - 127), exact; code 255 is NaN. */
static double ue8m0_value(uint8_t code)
{
    if (code == 0xFF)
        return NAN;
    return ldexp(1.0, (int)code - 127);
}

/* Nearest E4M3 code to y (a finite double), ties to the even code (the code's
 * last bit is the mantissa's last bit), magnitudes beyond 448 saturated to 448.
 * Found by comparing y with every finite non-negative E4M3 value. */
static uint8_t e4m3_nearest(double y)
{
    double mag = fabs(y);
    int best = 0;
    double best_err = INFINITY;
    if (mag >= 448.0) {
        best = 0x7E;
    } else {
        for (int c = 0; c <= 0x7E; ++c) {
            double err = fabs(e4m3_value((uint8_t)c) - mag);
            if (err < best_err || (err == best_err && (c & 1) == 0)) {
                best = c;
                best_err = err;
            }
        }
    }
    return (uint8_t)(signbit(y) ? (best | 0x80) : best);
}

/* Element (r, c) of op(X), X stored row-major with leading dimension ld. */
static double op_at(const uint16_t *X, int64_t ld, int trans, int64_t r, int64_t c)
{
    if (trans)
        return bf16_value(X[c * ld + r]);
    return bf16_value(X[r * ld + c]);
}

/* Element (i, j) of the input C, float32 or bf16. */
static double c_input(const void *C, int64_t ldc, int c_is_bf16, int64_t i, int64_t j)
{
    if (c_is_bf16)
        return bf16_value(((const uint16_t *)C)[i * ldc + j]);
    return (double)((const float *)C)[i * ldc + j];
}

/* One output element of GEMM. */
static void gemm_element(int64_t i, int64_t j, int64_t k, int transA, int transB, double alpha,
                         const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                         double beta, const void *C, int64_t ldc, int c_is_bf16,
                         double *ref, double *bound)
{
    double acc = 0.0, mag = 0.0;
    if (alpha != 0.0) {
        for (int64_t p = 0; p < k; ++p) {
            double prod = op_at(A, lda, transA, i, p) * op_at(B, ldb, transB, p, j);
            acc += prod;
            mag += fabs(prod);
        }
    }
    double value = alpha * acc;
    if (beta != 0.0)
        value += beta * c_input(C, ldc, c_is_bf16, i, j);
    *ref = value;
    *bound = mag;
}

/* One output element of SYRK: the product of rows i and j of op(A). */
static void syrk_element(int64_t i, int64_t j, int64_t k, int trans, double alpha,
                         const uint16_t *A, int64_t lda, double beta, const void *C,
                         int64_t ldc, int c_is_bf16, double *ref, double *bound)
{
    double acc = 0.0, mag = 0.0;
    if (alpha != 0.0) {
        for (int64_t p = 0; p < k; ++p) {
            double prod = op_at(A, lda, trans, i, p) * op_at(A, lda, trans, j, p);
            acc += prod;
            mag += fabs(prod);
        }
    }
    double value = alpha * acc;
    if (beta != 0.0)
        value += beta * c_input(C, ldc, c_is_bf16, i, j);
    *ref = value;
    *bound = mag;
}

/* One output element of the E4M3 GEMM: row i of A against row j of B. */
static void gemm_e4m3_element(int64_t i, int64_t j, int64_t k, double alpha, const uint8_t *A,
                              int64_t lda, const uint8_t *B, int64_t ldb, double beta,
                              const void *C, int64_t ldc, int c_is_bf16, double *ref,
                              double *bound)
{
    double acc = 0.0, mag = 0.0;
    if (alpha != 0.0) {
        for (int64_t p = 0; p < k; ++p) {
            double prod = e4m3_value(A[i * lda + p]) * e4m3_value(B[j * ldb + p]);
            acc += prod;
            mag += fabs(prod);
        }
    }
    double value = alpha * acc;
    if (beta != 0.0)
        value += beta * c_input(C, ldc, c_is_bf16, i, j);
    *ref = value;
    *bound = mag;
}

/* One output element of the MXFP8 GEMM: row i of A and row j of B, each element
 * times the scale of its group of 32 along K. */
static void gemm_mxfp8_element(int64_t i, int64_t j, int64_t k, double alpha, const uint8_t *A,
                               int64_t lda, const uint8_t *SA, int64_t ldsa, const uint8_t *B,
                               int64_t ldb, const uint8_t *SB, int64_t ldsb, double beta,
                               const void *C, int64_t ldc, int c_is_bf16, double *ref,
                               double *bound)
{
    double acc = 0.0, mag = 0.0;
    if (alpha != 0.0) {
        for (int64_t p = 0; p < k; ++p) {
            double a = e4m3_value(A[i * lda + p]) * ue8m0_value(SA[i * ldsa + p / 32]);
            double b = e4m3_value(B[j * ldb + p]) * ue8m0_value(SB[j * ldsb + p / 32]);
            double prod = a * b;
            acc += prod;
            mag += fabs(prod);
        }
    }
    double value = alpha * acc;
    if (beta != 0.0)
        value += beta * c_input(C, ldc, c_is_bf16, i, j);
    *ref = value;
    *bound = mag;
}

/* One output element of SYR2K: the two products of rows i and j of op(A), op(B). */
static void syr2k_element(int64_t i, int64_t j, int64_t k, int trans, double alpha, const uint16_t *A,
                          int64_t lda, const uint16_t *B, int64_t ldb, double beta, const void *C,
                          int64_t ldc, int c_is_bf16, double *ref, double *bound)
{
    double ab = 0.0, ba = 0.0, mag = 0.0;
    if (alpha != 0.0) {
        for (int64_t p = 0; p < k; ++p) {
            double x = op_at(A, lda, trans, i, p) * op_at(B, ldb, trans, j, p);
            double y = op_at(B, ldb, trans, i, p) * op_at(A, lda, trans, j, p);
            ab += x;
            ba += y;
            mag += fabs(x) + fabs(y);
        }
    }
    double value = alpha * (ab + ba);
    if (beta != 0.0)
        value += beta * c_input(C, ldc, c_is_bf16, i, j);
    *ref = value;
    *bound = mag;
}

/* Is (i, j) in the referenced triangle? uplo 0 = lower (i >= j), 1 = upper (i <= j). */
static int in_triangle(int uplo, int64_t i, int64_t j)
{
    return uplo == 0 ? (i >= j) : (i <= j);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for later parallel regions (host plumbing; no effect on any result). */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Full GEMM: ref and bound are m x n row-major with leading dimension ldr. */
void oracle_gemm(int64_t m, int64_t n, int64_t k, int transA, int transB, double alpha,
                 const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb, double beta,
                 const void *C, int64_t ldc, int c_is_bf16, double *ref, double *bound,
                 int64_t ldr)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < m; ++i)
        for (int64_t j = 0; j < n; ++j)
            gemm_element(i, j, k, transA, transB, alpha, A, lda, B, ldb, beta, C, ldc,
                         c_is_bf16, &ref[i * ldr + j], &bound[i * ldr + j]);
}

/* GEMM at `count` chosen positions (rows[t], cols[t]). */
void oracle_gemm_entries(int64_t k, int transA, int transB, double alpha, const uint16_t *A,
                         int64_t lda, const uint16_t *B, int64_t ldb, double beta, const void *C,
                         int64_t ldc, int c_is_bf16, int64_t count, const int64_t *rows,
                         const int64_t *cols, double *ref, double *bound)
{
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < count; ++t)
        gemm_element(rows[t], cols[t], k, transA, transB, alpha, A, lda, B, ldb, beta, C, ldc,
                     c_is_bf16, &ref[t], &bound[t]);
}

/* Full SYRK: entries outside the triangle are set to NaN (not referenced). */
void oracle_syrk(int uplo, int trans, int64_t n, int64_t k, double alpha, const uint16_t *A,
                 int64_t lda, double beta, const void *C, int64_t ldc, int c_is_bf16,
                 double *ref, double *bound, int64_t ldr)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < n; ++j) {
            if (in_triangle(uplo, i, j)) {
                syrk_element(i, j, k, trans, alpha, A, lda, beta, C, ldc, c_is_bf16,
                             &ref[i * ldr + j], &bound[i * ldr + j]);
            } else {
                ref[i * ldr + j] = NAN;
                bound[i * ldr + j] = NAN;
            }
        }
}

/* SYRK at chosen positions; positions outside the triangle give NaN. */
void oracle_syrk_entries(int uplo, int trans, int64_t k, double alpha, const uint16_t *A,
                         int64_t lda, double beta, const void *C, int64_t ldc, int c_is_bf16,
                         int64_t count, const int64_t *rows, const int64_t *cols, double *ref,
                         double *bound)
{
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < count; ++t) {
        if (in_triangle(uplo, rows[t], cols[t])) {
            syrk_element(rows[t], cols[t], k, trans, alpha, A, lda, beta, C, ldc, c_is_bf16,
                         &ref[t], &bound[t]);
        } else {
            ref[t] = NAN;
            bound[t] = NAN;
        }
    }
}

/* Full SYR2K: entries outside the triangle are set to NaN (not referenced). */
void oracle_syr2k(int uplo, int trans, int64_t n, int64_t k, double alpha, const uint16_t *A,
                  int64_t lda, const uint16_t *B, int64_t ldb, double beta, const void *C,
                  int64_t ldc, int c_is_bf16, double *ref, double *bound, int64_t ldr)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < n; ++j) {
            if (in_triangle(uplo, i, j)) {
                syr2k_element(i, j, k, trans, alpha, A, lda, B, ldb, beta, C, ldc, c_is_bf16,
                              &ref[i * ldr + j], &bound[i * ldr + j]);
            } else {
                ref[i * ldr + j] = NAN;
                bound[i * ldr + j] = NAN;
            }
        }
}

/* SYR2K at chosen positions; positions outside the triangle give NaN. */
void oracle_syr2k_entries(int uplo, int trans, int64_t k, double alpha, const uint16_t *A,
                          int64_t lda, const uint16_t *B, int64_t ldb, double beta, const void *C,
                          int64_t ldc, int c_is_bf16, int64_t count, const int64_t *rows,
                          const int64_t *cols, double *ref, double *bound)
{
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < count; ++t) {
        if (in_triangle(uplo, rows[t], cols[t])) {
            syr2k_element(rows[t], cols[t], k, trans, alpha, A, lda, B, ldb, beta, C, ldc,
                          c_is_bf16, &ref[t], &bound[t]);
        } else {
            ref[t] = NAN;
            bound[t] = NAN;
        }
    }
}

/* Full E4M3 GEMM C = alpha * A * B^T + beta * C; A [m, k], B [n, k]. */
void oracle_gemm_e4m3(int64_t m, int64_t n, int64_t k, double alpha, const uint8_t *A, int64_t lda,
                      const uint8_t *B, int64_t ldb, double beta, const void *C, int64_t ldc,
                      int c_is_bf16, double *ref, double *bound, int64_t ldr)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < m; ++i)
        for (int64_t j = 0; j < n; ++j)
            gemm_e4m3_element(i, j, k, alpha, A, lda, B, ldb, beta, C, ldc, c_is_bf16,
                              &ref[i * ldr + j], &bound[i * ldr + j]);
}

/* E4M3 GEMM at chosen positions. */
void oracle_gemm_e4m3_entries(int64_t k, double alpha, const uint8_t *A, int64_t lda,
                              const uint8_t *B, int64_t ldb, double beta, const void *C,
                              int64_t ldc, int c_is_bf16, int64_t count, const int64_t *rows,
                              const int64_t *cols, double *ref, double *bound)
{
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < count; ++t)
        gemm_e4m3_element(rows[t], cols[t], k, alpha, A, lda, B, ldb, beta, C, ldc, c_is_bf16,
                          &ref[t], &bound[t]);
}

/* Full MXFP8 GEMM C = alpha * (A . SA) * (B . SB)^T + beta * C; A [m, k], B [n, k]. */
void oracle_gemm_mxfp8(int64_t m, int64_t n, int64_t k, double alpha, const uint8_t *A, int64_t lda,
                       const uint8_t *SA, int64_t ldsa, const uint8_t *B, int64_t ldb,
                       const uint8_t *SB, int64_t ldsb, double beta, const void *C, int64_t ldc,
                       int c_is_bf16, double *ref, double *bound, int64_t ldr)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < m; ++i)
        for (int64_t j = 0; j < n; ++j)
            gemm_mxfp8_element(i, j, k, alpha, A, lda, SA, ldsa, B, ldb, SB, ldsb, beta, C, ldc,
                               c_is_bf16, &ref[i * ldr + j], &bound[i * ldr + j]);
}

/* MXFP8 GEMM at chosen positions. */
void oracle_gemm_mxfp8_entries(int64_t k, double alpha, const uint8_t *A, int64_t lda,
                               const uint8_t *SA, int64_t ldsa, const uint8_t *B, int64_t ldb,
                               const uint8_t *SB, int64_t ldsb, double beta, const void *C,
                               int64_t ldc, int c_is_bf16, int64_t count, const int64_t *rows,
                               const int64_t *cols, double *ref, double *bound)
{
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < count; ++t)
        gemm_mxfp8_element(rows[t], cols[t], k, alpha, A, lda, SA, ldsa, B, ldb, SB, ldsb, beta, C,
                           ldc, c_is_bf16, &ref[t], &bound[t]);
}

/* MXFP8 quantization of X [rows, k] (bf16 bits, leading dimension ldx) into E4M3
 * codes Q [rows, k] (ldq) and UE8M0 codes S [rows, ceil(k/32)] (lds), one per
 * group of 32 consecutive elements of a row (the last group may be shorter). */
void oracle_quantize_mxfp8(int64_t rows, int64_t k, const uint16_t *X, int64_t ldx, uint8_t *Q,
                           int64_t ldq, uint8_t *S, int64_t lds)
{
    int64_t groups = (k + 31) / 32;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t g = 0; g < groups; ++g) {
            int64_t p0 = 32 * g, p1 = p0 + 32 < k ? p0 + 32 : k;
            double amax = 0.0;
            int special = 0;
            for (int64_t p = p0; p < p1; ++p) {
                double x = bf16_value(X[i * ldx + p]);
                if (isnan(x) || isinf(x))
                    special = 1;
                else if (fabs(x) > amax)
                    amax = fabs(x);
            }
            if (special) {
                S[i * lds + g] = 0xFF;
                for (int64_t p = p0; p < p1; ++p)
                    Q[i * ldq + p] = 0x7F;
                continue;
            }
            int e = -127;
            if (amax > 0.0) {
                int ex;
                frexp(amax, &ex); /* amax = f * 2^ex, f in [0.5, 1): floor(log2(amax)) = ex - 1 */
                e = (ex - 1) - 8;
                if (e < -127)
                    e = -127;
                if (e > 127)
                    e = 127;
            }
            S[i * lds + g] = (uint8_t)(e + 127);
            for (int64_t p = p0; p < p1; ++p)
                Q[i * ldq + p] = e4m3_nearest(ldexp(bf16_value(X[i * ldx + p]), -e));
        }
}
