/*
 * Q4 group-64 matrix-vector product: plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this file's library.  It shares no code, header
 * or constant with the CUDA library it checks.
 *
 * What it computes is the plain definition of the decode matmul with the
 * dequantisation folded into the dot product (BaseRT: optimal LLM inference
 * on Apple Silicon with native Metal, §3.3 "Kernel fusion and
 * specialisation": each GEMV/GEMM dequantises inside its inner loop instead of
 * writing dequantised weights out; the result is the same as dequantising
 * first and then doing a dense product):
 *
 *     y[m][n] = sum_{k=0}^{K-1} ( s[n][k/64] * q[n][k] + b[n][k/64] ) * x[m][k]
 *
 * accumulated in fp64, in order k = 0 .. K-1.  It also returns
 *
 *     A[m][n] = sum_k | w[n][k] * x[m][k] |
 *
 * the scale of the per-element error bound.
 *
 * Storage: Wq uint32 [N][K/8]; code k of row n is bits 4*(k%8) .. 4*(k%8)+3
 * of word k/8 (lowest nibble first).  s, b, x are IEEE binary16 bit patterns;
 * they are converted exactly to fp64 by q4o_half_to_double below.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Test hook: Q4O_MUTANT selects a deliberately wrong variant so the pin tests
 * can show that each plausible mistake is caught.  0 = the real oracle. */
#ifndef Q4O_MUTANT
#define Q4O_MUTANT 0
#endif

/* IEEE 754 binary16 -> double, exact: 1 sign bit, 5 exponent bits (bias 15),
 * 10 fraction bits; exponent 0 is subnormal (f * 2^-24), 31 is inf/nan. */
double q4o_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25);
    return sign ? -v : v;
}

/* The 4-bit code of weight k in one packed row (the storage reading above:
 * lowest nibble first; the pages print no layout). */
int q4o_code(const uint32_t *row, int64_t k)
{
#if Q4O_MUTANT == 1 /* mistake: highest nibble first */
    return (int)((row[k / 8] >> (4 * (7 - k % 8))) & 0xFu);
#else
    return (int)((row[k / 8] >> (4 * (k % 8))) & 0xFu);
#endif
}

/* Dequantised weight w[n][k] = s * q + b, in fp64 (the affine group format
 * the BaseRT §3.3 kernels dequantise in their inner loop). */
static double q4o_weight(const uint32_t *row, const uint16_t *s_row, const uint16_t *b_row, int64_t k)
{
#if Q4O_MUTANT == 3 /* mistake: group of 32 instead of 64 */
    int64_t g = k / 32;
#else
    int64_t g = k / 64;
#endif
    double s = q4o_half_to_double(s_row[g]);
    double b = q4o_half_to_double(b_row[g]);
    double q = (double)q4o_code(row, k);
#if Q4O_MUTANT == 2 /* mistake: bias dropped */
    (void)b;
    return s * q;
#elif Q4O_MUTANT == 4 /* mistake: sign of the bias flipped */
    return s * q - b;
#else
    return s * q + b;
#endif
}

/*
 * The definition at the top of this file (BaseRT §3.3): y[m][i], A[m][i] for
 * the rows listed in rows[0..nrows) (all rows 0..N-1 when rows == NULL,
 * nrows = N), with x given in fp64: x [M][K], y and A [M][nrows].  A may be
 * NULL.  nthreads <= 0 uses the OpenMP default.  Returns 0, or -1 on a bad
 * argument.
 */
int q4o_gemv_f64(const uint32_t *Wq, const uint16_t *scales, const uint16_t *biases,
                 const double *xd, int64_t M, int64_t N, int64_t K,
                 const int64_t *rows, int64_t nrows, double *y, double *A, int nthreads)
{
    if (!Wq || !scales || !biases || !xd || !y || M < 1 || N < 0 || K < 64 || K % 64)
        return -1;
    if (!rows)
        nrows = N;
    int64_t words = K / 8, groups = K / 64;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads)
#endif
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t n = rows ? rows[i] : i;
        const uint32_t *row = Wq + n * words;
        const uint16_t *s_row = scales + n * groups;
        const uint16_t *b_row = biases + n * groups;
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
#if Q4O_MUTANT == 5 /* mistake: transposed operand (x indexed by the row) */
                double xv = xd[m * K + (n % K)];
#else
                double xv = xd[m * K + k];
#endif
                double t = q4o_weight(row, s_row, b_row, k) * xv;
                acc += t;
                mag += fabs(t);
            }
            y[m * nrows + i] = acc;
            if (A)
                A[m * nrows + i] = mag;
        }
    }
    return 0;
}

/* Same with x given as fp16 bit patterns (converted exactly to fp64). */
int q4o_gemv(const uint32_t *Wq, const uint16_t *scales, const uint16_t *biases,
             const uint16_t *x, int64_t M, int64_t N, int64_t K,
             const int64_t *rows, int64_t nrows, double *y, double *A, int nthreads)
{
    if (!x || M < 1 || K < 64)
        return -1;
    double *xd = (double *)malloc(sizeof(double) * (size_t)(M * K));
    if (!xd)
        return -1;
    for (int64_t i = 0; i < M * K; ++i)
        xd[i] = q4o_half_to_double(x[i]);
    int rc = q4o_gemv_f64(Wq, scales, biases, xd, M, N, K, rows, nrows, y, A, nthreads);
    free(xd);
    return rc;
}

/*
 * The same product for 8-bit codes (the pages' 8-bit format: BaseRT §3.3 and
 * §4.1 evaluate Q4 and Q8; the bit layout is not printed, so the one the
 * library fixes is used): Wq uint32 [N][K/4]; code k of row n is bits
 * 8*(k%4) .. 8*(k%4)+7 of word k/4 (lowest byte first), q in 0..255; one fp16
 * scale and bias per group of 64; w = s * q + b; fp64 accumulation in order
 * k = 0 .. K-1, and A = sum_k |w x| as above.
 */
int q8o_code(const uint32_t *row, int64_t k)
{
#if Q4O_MUTANT == 6 /* mistake: highest byte first */
    return (int)((row[k / 4] >> (8 * (3 - k % 4))) & 0xFFu);
#elif Q4O_MUTANT == 7 /* mistake: only the low nibble of each byte */
    return (int)((row[k / 4] >> (8 * (k % 4))) & 0x0Fu);
#else
    return (int)((row[k / 4] >> (8 * (k % 4))) & 0xFFu);
#endif
}

int q8o_gemv_f64(const uint32_t *Wq, const uint16_t *scales, const uint16_t *biases,
                 const double *xd, int64_t M, int64_t N, int64_t K,
                 const int64_t *rows, int64_t nrows, double *y, double *A, int nthreads)
{
    if (!Wq || !scales || !biases || !xd || !y || M < 1 || N < 0 || K < 64 || K % 64)
        return -1;
    if (!rows)
        nrows = N;
    int64_t words = K / 4, groups = K / 64;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads)
#endif
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t n = rows ? rows[i] : i;
        const uint32_t *row = Wq + n * words;
        const uint16_t *s_row = scales + n * groups;
        const uint16_t *b_row = biases + n * groups;
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
#if Q4O_MUTANT == 8 /* mistake: group of 32 instead of 64 (clamped to stay in the row) */
                int64_t g = k / 32 < groups ? k / 32 : groups - 1;
#else
                int64_t g = k / 64;
#endif
                double w = q4o_half_to_double(s_row[g]) * (double)q8o_code(row, k) + q4o_half_to_double(b_row[g]);
                double t = w * xd[m * K + k];
                acc += t;
                mag += fabs(t);
            }
            y[m * nrows + i] = acc;
            if (A)
                A[m * nrows + i] = mag;
        }
    }
    return 0;
}

int q8o_gemv(const uint32_t *Wq, const uint16_t *scales, const uint16_t *biases,
             const uint16_t *x, int64_t M, int64_t N, int64_t K,
             const int64_t *rows, int64_t nrows, double *y, double *A, int nthreads)
{
    if (!x || M < 1 || K < 64)
        return -1;
    double *xd = (double *)malloc(sizeof(double) * (size_t)(M * K));
    if (!xd)
        return -1;
    for (int64_t i = 0; i < M * K; ++i)
        xd[i] = q4o_half_to_double(x[i]);
    int rc = q8o_gemv_f64(Wq, scales, biases, xd, M, N, K, rows, nrows, y, A, nthreads);
    free(xd);
    return rc;
}

/* b-bit codes, b in 2..8 (BaseRT §3.3 and §4.1: dedicated kernels per
 * quantisation format, 2- to 8-bit): code k of a row occupies bits
 * b*k .. b*k+b-1 of the row's little-endian bit stream, i.e. of its uint32
 * words taken lowest bit first, a code crossing a word boundary continuing in
 * the low bits of the next word.  For b = 4 and 8 this is the layout above. */
int qbo_code(const uint32_t *row, int64_t k, int bits)
{
#if Q4O_MUTANT == 9 /* mistake: codes packed one bit further on */
    int64_t p = (int64_t)bits * k + 1;
#else
    int64_t p = (int64_t)bits * k;
#endif
    int64_t w = p / 32;
    int sh = (int)(p % 32);
    uint64_t v = row[w] >> sh;
#if Q4O_MUTANT == 10 /* mistake: a code crossing a word boundary loses its high bits */
    (void)0;
#else
    if (sh + bits > 32)
        v |= (uint64_t)row[w + 1] << (32 - sh);
#endif
    return (int)(v & ((1u << bits) - 1u));
}

int qbo_gemv_f64(const uint32_t *Wq, const uint16_t *scales, const uint16_t *biases,
                 const double *xd, int64_t M, int64_t N, int64_t K, int bits,
                 const int64_t *rows, int64_t nrows, double *y, double *A, int nthreads)
{
    if (!Wq || !scales || !biases || !xd || !y || M < 1 || N < 0 || K < 64 || K % 64 || bits < 2 || bits > 8)
        return -1;
    if (!rows)
        nrows = N;
    int64_t words = K * bits / 32, groups = K / 64;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads)
#endif
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t n = rows ? rows[i] : i;
        const uint32_t *row = Wq + n * words;
        const uint16_t *s_row = scales + n * groups;
        const uint16_t *b_row = biases + n * groups;
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
#if Q4O_MUTANT == 9
                /* the shifted stream runs one bit past the last code: clamp to stay in the row */
                int c = k == K - 1 ? qbo_code(row, k - 1, bits) : qbo_code(row, k, bits);
#else
                int c = qbo_code(row, k, bits);
#endif
                int64_t g = k / 64;
                double w = q4o_half_to_double(s_row[g]) * (double)c + q4o_half_to_double(b_row[g]);
                double t = w * xd[m * K + k];
                acc += t;
                mag += fabs(t);
            }
            y[m * nrows + i] = acc;
            if (A)
                A[m * nrows + i] = mag;
        }
    }
    return 0;
}

int qbo_gemv(const uint32_t *Wq, const uint16_t *scales, const uint16_t *biases,
             const uint16_t *x, int64_t M, int64_t N, int64_t K, int bits,
             const int64_t *rows, int64_t nrows, double *y, double *A, int nthreads)
{
    if (!x || M < 1 || K < 64)
        return -1;
    double *xd = (double *)malloc(sizeof(double) * (size_t)(M * K));
    if (!xd)
        return -1;
    for (int64_t i = 0; i < M * K; ++i)
        xd[i] = q4o_half_to_double(x[i]);
    int rc = qbo_gemv_f64(Wq, scales, biases, xd, M, N, K, bits, rows, nrows, y, A, nthreads);
    free(xd);
    return rc;
}

/* Number of OpenMP threads this library would use by default (1 without OpenMP). */
int q4o_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
