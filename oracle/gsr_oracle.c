/*
 * gsr_oracle.c - plain CPU oracle for the fused operator
 *
 *     C[m,n] = ReLU( alpha * sum_{k=0}^{K-1} A[m,k] * B[k,n] )
 *
 * with A (M,K) and B (K,N) row-major IEEE binary16, the sum carried in fp64
 * and C rounded once to binary16.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker for the GPU library, not
 * part of it: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg may load it.  It shares no code, header, table or constant with
 * the CUDA path.  It is deliberately slow and unblocked so that a reader can
 * check it against the definition by eye.
 *
 * Sources (page title and section):
 *  - "Tutorial14: 使用TileLang语言编写attention算子" (PKUHPC scow-tutorial),
 *    section 3 (算子介绍), the operator formula: C = ReLU((sum_k A*B) * alpha),
 *    ReLU(x) = max(x, 0).  Section 2 (编写算子), the gemm_fused kernel: inputs
 *    float16, accumulator "float" (wider than the inputs), the accumulator is
 *    multiplied by the float32 scale first and the max with 0 comes second,
 *    then the result is written out as float16.
 *  - "TileKernels：面向大语言模型的高性能GPU算子库解析", section 五 (开发实践指南),
 *    the custom_matmul example: the plain triple loop acc = 0; acc += A*B;
 *    C = acc, which is the shape of the loop below.
 *
 * Readings where the pages are silent:
 *  - the float32 -> float16 conversion of the result rounds to nearest, ties
 *    to even (IEEE 754 default); here it is applied once, to the fp64 value;
 *  - magnitudes past the binary16 range become infinity; subnormals are kept;
 *  - ReLU maps -0.0 and NaN to +0.0 (x > 0 ? x : 0), the same answer a
 *    max(x, 0) with IEEE maxNum semantics gives;
 *  - K == 0 is an empty sum, so every output is ReLU(alpha * 0) = +0.
 *
 * The loop order is i, k, n: for one output row, acc[n] collects the products
 * in increasing k, which is exactly the summation order of the textbook
 * i, n, k loop.  Each product of two binary16 values is exact in fp64
 * (11 x 11 significand bits), so only the running sum rounds.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared -fopenmp
 * (no fast-math; the default round-to-nearest mode is assumed by rint()).
 */
#define _DEFAULT_SOURCE
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- IEEE 754 binary16 codec, written from the format's definition ------ */

/* binary16 bit pattern -> exact double.
 * Fields: sign (1 bit), biased exponent e (5 bits, bias 15), fraction f
 * (10 bits).  e == 0: subnormal, value f * 2^-24.  e == 31: infinity (f == 0)
 * or NaN.  Otherwise (1024 + f) * 2^(e - 25) = (1 + f/1024) * 2^(e - 15). */
double oracle_f16_decode(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -24);
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + f), e - 25);
    return sign ? -mag : mag;
}

/* double -> binary16 bit pattern, rounding to nearest with ties to even.
 * Below 2^-14 the representable values are the multiples of 2^-24, so the
 * scaled value a * 2^24 is rounded to an integer (a result of 1024 is the
 * smallest normal, whose bit pattern is also 1024).  At or above 2^-14 the
 * significand is scaled into [1024, 2048] for the quantum 2^(E-10), rounded,
 * and a carry to 2048 bumps the exponent; exponents past 15 overflow to
 * infinity.  The scalings are by powers of two, hence exact, so rint() makes
 * the only rounding. */
uint16_t oracle_f16_encode(double x)
{
    if (isnan(x))
        return 0x7e00;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isinf(a))
        return sign | 0x7c00;
    if (a < ldexp(1.0, -14)) {
        double q = rint(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)q);
    }
    int ex;
    (void)frexp(a, &ex);          /* a = m * 2^ex, 0.5 <= m < 1 */
    int E = ex - 1;               /* a = 1.xxx * 2^E */
    double q = rint(ldexp(a, 10 - E));
    if (q == 2048.0) {
        q = 1024.0;
        E += 1;
    }
    if (E > 15)
        return sign | 0x7c00;
    return (uint16_t)(sign | (uint16_t)(((E + 15) << 10) | ((int)q - 1024)));
}

void oracle_f16_decode_array(const uint16_t *h, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f16_decode(h[i]);
}

void oracle_f16_encode_array(const double *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f16_encode(x[i]);
}

/* ---- the operator --------------------------------------------------------- */

static double g_dec[65536];
static int g_dec_ready;

static void build_decode_table(void)
{
    if (g_dec_ready)
        return;
    for (int i = 0; i < 65536; ++i)
        g_dec[i] = oracle_f16_decode((uint16_t)i);
    g_dec_ready = 1;
}

/* C (and optionally Z) for the requested output rows.
 *
 *   A      (M, K) binary16 bit patterns, row-major.
 *   B      (K, N) binary16 bit patterns, row-major.
 *   C      output, (R, N) binary16 bit patterns, row-major.
 *   Z      optional output, (R, N) doubles: alpha * sum, before the ReLU.
 *   rows   optional list of R row indices in [0, M); NULL means all M rows
 *          in order (R = M).  Output row r holds input row rows[r].
 *
 * Returns 0 on success, -1 on a bad argument, -2 when out of memory. */
int oracle_gemm_scale_relu(const uint16_t *A, const uint16_t *B, uint16_t *C,
                           double *Z, int64_t M, int64_t N, int64_t K,
                           float alpha, const int64_t *rows, int64_t nrows)
{
    if (M < 0 || N < 0 || K < 0)
        return -1;
    int64_t R = rows ? nrows : M;
    if (R < 0)
        return -1;
    if (rows)
        for (int64_t r = 0; r < R; ++r)
            if (rows[r] < 0 || rows[r] >= M)
                return -1;
    if (R == 0 || N == 0)
        return 0;
    if (!C || (K > 0 && (!A || !B)))
        return -1;
    build_decode_table();

    const double alpha_d = (double)alpha;   /* float32 -> double is exact */
    int failed = 0;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < R; ++r) {
        int64_t i = rows ? rows[r] : r;
        double *acc = (double *)calloc((size_t)N, sizeof(double));
        if (!acc) {
#pragma omp atomic write
            failed = 1;
            continue;
        }
        for (int64_t k = 0; k < K; ++k) {
            double a = g_dec[A[i * K + k]];
            const uint16_t *brow = B + k * N;
            for (int64_t n = 0; n < N; ++n)
                acc[n] += a * g_dec[brow[n]];
        }
        for (int64_t n = 0; n < N; ++n) {
            double z = alpha_d * acc[n];           /* scale first ...  */
            double y = z > 0.0 ? z : 0.0;          /* ... then ReLU    */
            if (Z)
                Z[r * N + n] = z;
            C[r * N + n] = oracle_f16_encode(y);
        }
        free(acc);
    }
    return failed ? -2 : 0;
}

/* ---- further epilogues on the same sum -------------------------------------
 *
 * kind 0: ReLU(alpha * sum)               (same result as oracle_gemm_scale_relu)
 * kind 1: alpha * sum                      (the plain tiled GEMM when alpha == 1: the
 *                                           make_matmul section of the aikraft.ru TileLang
 *                                           tutorial survey, "Тилированное умножение матриц")
 * kind 2: GELU(sum + bias[n])              (its make_matmul_bias_gelu section, "Слияние
 *                                           эпиколов: GEMM + Bias + GELU": bias added, then
 *                                           a GELU approximation written with an exponential)
 *
 * GELU reading: the tanh approximation 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))),
 * written through the exponential as x / (1 + exp(-2u)) with u = sqrt(2/pi)(x + 0.044715 x^3)
 * (the same function, since 1 + tanh(u) = 2 / (1 + exp(-2u)); this form has no cancellation
 * for large negative x).  bias holds N
 * binary16 values (ignored unless kind == 2).  Y (optional) receives the fp64 value that
 * is rounded into C.  Rows as for oracle_gemm_scale_relu.  Returns 0, -1 (bad argument)
 * or -2 (out of memory). */
static double gelu_exp_form(double x)
{
    const double u = sqrt(2.0 / M_PI) * (x + 0.044715 * x * x * x);
    return x / (1.0 + exp(-2.0 * u));
}

int oracle_gemm_epilogue(const uint16_t *A, const uint16_t *B, const uint16_t *bias,
                         uint16_t *C, double *Y, int64_t M, int64_t N, int64_t K,
                         float alpha, int kind, const int64_t *rows, int64_t nrows)
{
    if (M < 0 || N < 0 || K < 0 || kind < 0 || kind > 2)
        return -1;
    int64_t R = rows ? nrows : M;
    if (R < 0)
        return -1;
    if (rows)
        for (int64_t r = 0; r < R; ++r)
            if (rows[r] < 0 || rows[r] >= M)
                return -1;
    if (R == 0 || N == 0)
        return 0;
    if (!C || (K > 0 && (!A || !B)) || (kind == 2 && !bias))
        return -1;
    build_decode_table();

    const double alpha_d = (double)alpha;
    int failed = 0;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < R; ++r) {
        int64_t i = rows ? rows[r] : r;
        double *acc = (double *)calloc((size_t)N, sizeof(double));
        if (!acc) {
#pragma omp atomic write
            failed = 1;
            continue;
        }
        for (int64_t k = 0; k < K; ++k) {
            double a = g_dec[A[i * K + k]];
            const uint16_t *brow = B + k * N;
            for (int64_t n = 0; n < N; ++n)
                acc[n] += a * g_dec[brow[n]];
        }
        for (int64_t n = 0; n < N; ++n) {
            double y;
            if (kind == 0) {
                double z = alpha_d * acc[n];
                y = z > 0.0 ? z : 0.0;
            } else if (kind == 1) {
                y = alpha_d * acc[n];
            } else {
                y = gelu_exp_form(acc[n] + g_dec[bias[n]]);
            }
            if (Y)
                Y[r * N + n] = y;
            C[r * N + n] = oracle_f16_encode(y);
        }
        free(acc);
    }
    return failed ? -2 : 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
