/*
 * gemm_oracle.c -- plain, slow CPU oracle for row-major dense GEMM
 *
 *     C = alpha * A * B + beta * C
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg load this library. The GPU library never links,
 * includes or calls it, and the two share no source.
 *
 * What is computed (the definition, restated in plain loops):
 *
 *     for every i < M, j < N:
 *         acc    = sum over k < K of A[i,k] * B[k,j]
 *         C[i,j] = alpha * acc + beta * C[i,j]
 *
 *   - "Sgemm [128,128,8]" (jianshu page): the comment above the kernel defines
 *     gemm as C = alpha*A*B + beta*C with every matrix stored row-major, and the
 *     page's host reference routine host_gemm is exactly this loop nest with the
 *     alpha/beta update applied once per output element.
 *   - "CUDA学习之路[11]：矩阵乘法计算详解" (dlog page), section 什么是矩阵乘法
 *     ("what is a matrix multiply"): the CPU sgemm triple loop, sum over k of
 *     A[i*K+k] * B[k*N+j].
 *   - C++ warp-matrix-function (WMMA) page, type table: __half and
 *     __nv_bfloat16 inputs accumulate into float; signed char and unsigned char
 *     inputs accumulate into int; __half inputs may also produce a __half
 *     result; precision::tf32 inputs accumulate into float; double inputs
 *     accumulate into double.
 *
 * Row-major with leading dimensions: element (i,j) of X sits at X[i*ldx + j]
 * ("Sgemm [128,128,8]", the A(i,j)/B(i,j)/C(i,j) index macros).
 *
 * Precision.
 *   - Floating inputs (fp32, bf16, fp16) are first decoded exactly to double.
 *     Their products carry at most 24+24 significant bits, so every product is
 *     exact in double; the K-term sum is accumulated in double, one rounding per
 *     add, in increasing k. The result is returned as double, not rounded to
 *     fp32.
 *   - int8 inputs accumulate exactly in int64. The alpha/beta update is taken
 *     modulo 2^64 in unsigned arithmetic and the low 32 bits are returned as a
 *     two's-complement int32: that is int32 wrap-around arithmetic, which is what
 *     an int32 accumulator and int32 output imply when a result overflows.
 *   - double inputs (oracle_gemm_f64 called directly): products and sums are
 *     rounded in double, so this reference is exactly as precise as a double
 *     GPU kernel; the fp64 comparison is graded with a tolerance derived from
 *     that rounding instead of bit for bit.
 *   - 16-bit results (the table's half -> half row, and its bf16 analogue):
 *     the result is computed exactly as above (in double) and then rounded
 *     once to the 16-bit format, round-to-nearest, ties to even. The GPU
 *     accumulates in fp32; the accumulator width the page lists for this row
 *     (half) is a hardware detail with no fixed summation order, so the
 *     definition used here is "the exact product, rounded once".
 *   - tf32 inputs: each fp32 value is reduced to tf32 (8 exponent bits, 10
 *     fraction bits) by clearing its 13 lowest fraction bits, i.e. truncation
 *     toward zero; the reduced values are then multiplied exactly as above.
 *     The page names the tf32 precision but not how an fp32 value becomes one;
 *     truncation is the reading taken here.
 *
 * Readings where the pages are silent:
 *   - beta == 0: C is not read (BLAS convention), so NaN/Inf in C do not
 *     propagate. The jianshu kernel always reads C; the tiled-multiply page and
 *     the dlog kernels never read it. The plain definition with "beta*C" taken
 *     as the zero term when beta is zero is the reading used here.
 *   - alpha == 0: the product is still formed and multiplied by zero.
 *   - K == 0: acc is the empty sum 0, so C = beta*C.
 *   - M == 0 or N == 0: nothing is written.
 *
 * Loop order is i-k-j. Each C[i,j] still receives its terms in increasing k
 * with one rounding per add, exactly as in the textbook i-j-k loop; only the
 * order in which different (i,j) are visited changes, so the result is the same
 * bit for bit. Rows are independent and are spread over OpenMP threads when the
 * library is built with OpenMP; the thread count does not change the result.
 * Build without -ffast-math and with -ffp-contract=off so that no add or
 * multiply is fused or reassociated.
 *
 * Return value of every entry point: 0 on success, -1 for a negative size or a
 * leading dimension smaller than the row length, -2 when scratch memory cannot
 * be allocated.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- decoders */

/* bf16 is the upper half of an IEEE binary32 pattern. */
double oracle_decode_bf16(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24); /* subnormal: m * 2^(1-15-10) */
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* ---------------------------------------------------------------- encoders */

/*
 * Rounds x to the nearest value of a binary format with `ebits` exponent bits
 * (bias 2^(ebits-1) - 1) and `mbits` stored fraction bits, ties to even, and
 * returns its bit pattern: gradual underflow below the smallest normal, +-Inf
 * past the largest finite value plus half a unit in its last place, a quiet
 * NaN for NaN. Works on the value, not on the bits of x: the quantum (the
 * spacing of the target format near |x|) is a power of two, so |x| / quantum
 * is exact and only the final integer rounding decides.
 */
static uint32_t encode_binary(double x, int ebits, int mbits)
{
    const int bias = (1 << (ebits - 1)) - 1;
    const int emin = 1 - bias; /* exponent of the smallest normal */
    const uint32_t sign = signbit(x) ? 1u : 0u;
    const uint32_t sign_bit = sign << (ebits + mbits);
    const uint32_t exp_all = ((1u << ebits) - 1u) << mbits;
    if (isnan(x)) return exp_all | (1u << (mbits - 1)); /* quiet NaN */
    double a = fabs(x);
    if (isinf(a)) return sign_bit | exp_all;
    if (a == 0.0) return sign_bit;
    int e;
    frexp(a, &e); /* a = f * 2^e, f in [0.5, 1): floor(log2 a) = e - 1 */
    int ex = e - 1;
    if (ex < emin) ex = emin; /* subnormal range: fixed quantum */
    const double quantum = ldexp(1.0, ex - mbits);
    const double q = a / quantum; /* exact */
    double r = floor(q);
    const double frac = q - r;     /* exact */
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    /* r * quantum is the rounded magnitude; r may have carried to 2^(mbits+1). */
    double v = r * quantum;
    const double max_finite = ldexp(2.0 - ldexp(1.0, -mbits), bias);
    if (v > max_finite) return sign_bit | exp_all;
    if (v < ldexp(1.0, emin)) /* subnormal: fraction = v / 2^(emin - mbits) */
        return sign_bit | (uint32_t)ldexp(v, -(emin - mbits));
    frexp(v, &e);
    ex = e - 1;
    const uint32_t frac_bits = (uint32_t)(ldexp(v, mbits - ex) - ldexp(1.0, mbits));
    return sign_bit | ((uint32_t)(ex + bias) << mbits) | frac_bits;
}

uint16_t oracle_encode_f16(double x) { return (uint16_t)encode_binary(x, 5, 10); }
uint16_t oracle_encode_bf16(double x) { return (uint16_t)encode_binary(x, 8, 7); }

/* fp32 -> tf32 as read above: the 13 lowest fraction bits cleared. */
float oracle_round_tf32(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    u &= ~0x1fffu;
    memcpy(&x, &u, sizeof x);
    return x;
}

/* ------------------------------------------------------------ double core */

static int bad_shape(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                     int64_t ldc)
{
    if (M < 0 || N < 0 || K < 0) return 1;
    if (M > 0 && K > 0 && lda < K) return 1;
    if (K > 0 && N > 0 && ldb < N) return 1;
    if (M > 0 && N > 0 && ldc < N) return 1;
    return 0;
}

/*
 * The definition in double. A is M x K (row stride lda), B is K x N (row stride
 * ldb), C is M x N (row stride ldc) and holds C0 on entry.
 */
int oracle_gemm_f64(int64_t M, int64_t N, int64_t K, double alpha,
                    const double *A, int64_t lda, const double *B, int64_t ldb,
                    double beta, double *C, int64_t ldc)
{
    if (bad_shape(M, N, K, lda, ldb, ldc)) return -1;
    if (M == 0 || N == 0) return 0;
    int status = 0;
#pragma omp parallel
    {
        double *acc = (double *)malloc(sizeof(double) * (size_t)N);
        if (!acc) {
#pragma omp atomic write
            status = -2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < M; i++) {
                for (int64_t j = 0; j < N; j++) acc[j] = 0.0;
                for (int64_t k = 0; k < K; k++) {
                    double a = A[i * lda + k];
                    const double *brow = B + k * ldb;
                    for (int64_t j = 0; j < N; j++) acc[j] += a * brow[j];
                }
                double *crow = C + i * ldc;
                for (int64_t j = 0; j < N; j++) {
                    double scaled = alpha * acc[j];
                    crow[j] = (beta == 0.0) ? scaled : scaled + beta * crow[j];
                }
            }
            free(acc);
        }
    }
    return status;
}

/* ------------------------------------------------- typed float entry points */

/*
 * Each typed entry point decodes A and B exactly into dense double copies (the
 * values the GPU sees, nothing rounded), reads C0 from the double array C, and
 * runs the double core. C (double, row stride ldc) holds C0 on entry and the
 * unrounded result on exit.
 */
typedef double (*decode_fn)(const void *base, int64_t idx);

static double dec_f32(const void *p, int64_t i) { return (double)((const float *)p)[i]; }
static double dec_bf16(const void *p, int64_t i) { return oracle_decode_bf16(((const uint16_t *)p)[i]); }
static double dec_f16(const void *p, int64_t i) { return oracle_decode_f16(((const uint16_t *)p)[i]); }
static double dec_tf32(const void *p, int64_t i)
{
    return (double)oracle_round_tf32(((const float *)p)[i]);
}

static int typed_gemm(decode_fn dec, int64_t M, int64_t N, int64_t K,
                      double alpha, const void *A, int64_t lda, const void *B,
                      int64_t ldb, double beta, double *C, int64_t ldc)
{
    if (bad_shape(M, N, K, lda, ldb, ldc)) return -1;
    if (M == 0 || N == 0) return 0;
    double *a = (double *)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    double *b = (double *)malloc(sizeof(double) * (size_t)(K * N > 0 ? K * N : 1));
    if (!a || !b) {
        free(a);
        free(b);
        return -2;
    }
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; i++)
        for (int64_t k = 0; k < K; k++) a[i * K + k] = dec(A, i * lda + k);
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < K; k++)
        for (int64_t j = 0; j < N; j++) b[k * N + j] = dec(B, k * ldb + j);
    int st = oracle_gemm_f64(M, N, K, alpha, a, K, b, N, beta, C, ldc);
    free(a);
    free(b);
    return st;
}

int oracle_gemm_f32(int64_t M, int64_t N, int64_t K, double alpha,
                    const float *A, int64_t lda, const float *B, int64_t ldb,
                    double beta, double *C, int64_t ldc)
{
    return typed_gemm(dec_f32, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc);
}

int oracle_gemm_bf16(int64_t M, int64_t N, int64_t K, double alpha,
                     const uint16_t *A, int64_t lda, const uint16_t *B,
                     int64_t ldb, double beta, double *C, int64_t ldc)
{
    return typed_gemm(dec_bf16, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc);
}

int oracle_gemm_f16(int64_t M, int64_t N, int64_t K, double alpha,
                    const uint16_t *A, int64_t lda, const uint16_t *B,
                    int64_t ldb, double beta, double *C, int64_t ldc)
{
    return typed_gemm(dec_f16, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc);
}

/* tf32 inputs: fp32 A and B reduced to tf32, then the exact product. */
int oracle_gemm_tf32(int64_t M, int64_t N, int64_t K, double alpha,
                     const float *A, int64_t lda, const float *B, int64_t ldb,
                     double beta, double *C, int64_t ldc)
{
    return typed_gemm(dec_tf32, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc);
}

/*
 * 16-bit inputs and a 16-bit C of the same format (is_bf16 selects bf16, else
 * IEEE binary16): C holds the 16-bit C0 on entry (not read when beta == 0) and
 * on exit round_to_16(alpha * sum_k A[i,k] B[k,j] + beta * C0[i,j]), the
 * right-hand side evaluated in double as in the other entry points.
 */
static int gemm_out16(int is_bf16, int64_t M, int64_t N, int64_t K, double alpha,
                      const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                      double beta, uint16_t *C, int64_t ldc)
{
    if (bad_shape(M, N, K, lda, ldb, ldc)) return -1;
    if (M == 0 || N == 0) return 0;
    double *c = (double *)malloc(sizeof(double) * (size_t)(M * N));
    if (!c) return -2;
    for (int64_t i = 0; i < M; i++)
        for (int64_t j = 0; j < N; j++)
            c[i * N + j] = (beta == 0.0) ? 0.0
                           : is_bf16     ? oracle_decode_bf16(C[i * ldc + j])
                                         : oracle_decode_f16(C[i * ldc + j]);
    int st = typed_gemm(is_bf16 ? dec_bf16 : dec_f16, M, N, K, alpha, A, lda, B, ldb, beta, c,
                        N);
    if (st == 0)
        for (int64_t i = 0; i < M; i++)
            for (int64_t j = 0; j < N; j++)
                C[i * ldc + j] = is_bf16 ? oracle_encode_bf16(c[i * N + j])
                                         : oracle_encode_f16(c[i * N + j]);
    free(c);
    return st;
}

int oracle_gemm_f16_f16(int64_t M, int64_t N, int64_t K, double alpha,
                        const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                        double beta, uint16_t *C, int64_t ldc)
{
    return gemm_out16(0, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc);
}

int oracle_gemm_bf16_bf16(int64_t M, int64_t N, int64_t K, double alpha,
                          const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                          double beta, uint16_t *C, int64_t ldc)
{
    return gemm_out16(1, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc);
}

/* ------------------------------------------------------------------- int8 */

/*
 * 8-bit integer inputs (signed char, or unsigned char when is_unsigned), int64
 * accumulation, int32 output with wrap-around. C holds the int32 C0 on entry
 * (not read when beta == 0) and the result on exit.
 */
static int int8_gemm(int is_unsigned, int64_t M, int64_t N, int64_t K, int32_t alpha,
                     const void *A8, int64_t lda, const void *B8, int64_t ldb, int32_t beta,
                     int32_t *C, int64_t ldc)
{
    const int8_t *As = (const int8_t *)A8, *Bs = (const int8_t *)B8;
    const uint8_t *Au = (const uint8_t *)A8, *Bu = (const uint8_t *)B8;
    if (bad_shape(M, N, K, lda, ldb, ldc)) return -1;
    if (M == 0 || N == 0) return 0;
    int status = 0;
#pragma omp parallel
    {
        int64_t *acc = (int64_t *)malloc(sizeof(int64_t) * (size_t)N);
        if (!acc) {
#pragma omp atomic write
            status = -2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < M; i++) {
                for (int64_t j = 0; j < N; j++) acc[j] = 0;
                for (int64_t k = 0; k < K; k++) {
                    const int64_t a = is_unsigned ? (int64_t)Au[i * lda + k]
                                                  : (int64_t)As[i * lda + k];
                    for (int64_t j = 0; j < N; j++) {
                        const int64_t b = is_unsigned ? (int64_t)Bu[k * ldb + j]
                                                      : (int64_t)Bs[k * ldb + j];
                        acc[j] += a * b;
                    }
                }
                int32_t *crow = C + i * ldc;
                for (int64_t j = 0; j < N; j++) {
                    uint64_t v = (uint64_t)(int64_t)alpha * (uint64_t)acc[j];
                    if (beta != 0)
                        v += (uint64_t)(int64_t)beta * (uint64_t)(int64_t)crow[j];
                    uint32_t low = (uint32_t)v; /* keep the low 32 bits */
                    int32_t out;
                    memcpy(&out, &low, sizeof out); /* two's complement view */
                    crow[j] = out;
                }
            }
            free(acc);
        }
    }
    return status;
}

int oracle_gemm_s8(int64_t M, int64_t N, int64_t K, int32_t alpha,
                   const int8_t *A, int64_t lda, const int8_t *B, int64_t ldb,
                   int32_t beta, int32_t *C, int64_t ldc)
{
    return int8_gemm(0, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc);
}

/* unsigned char inputs (the WMMA table's unsigned char -> int row). */
int oracle_gemm_u8(int64_t M, int64_t N, int64_t K, int32_t alpha,
                   const uint8_t *A, int64_t lda, const uint8_t *B, int64_t ldb,
                   int32_t beta, int32_t *C, int64_t ldc)
{
    return int8_gemm(1, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc);
}

/* Threads the oracle will use (1 when built without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
