/*
 * Dense GEMM oracle: C = A . B computed the plain way, in double precision.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark load it.  It shares no source with the CUDA path.
 *
 * What it computes follows "Shared memory and tensor cores" (ml-compiler-from-
 * scratch ch. 13), section 13.1: a GEMM C = A @ B is 2*M*N*K floating-point
 * operations, one multiply and one add per (i, j, k) triple, and nothing else.
 * Section 13.8 of the same page fixes the precision contract of the tensor-core
 * paths: products of the narrow inputs are formed exactly and summed in FP32.
 * This oracle is stricter: every product of two FP32, BF16 or FP16 values is
 * exact in IEEE double (at most 24 + 24 significand bits < 53), and the sums are done in double,
 * so the only rounding is that of a double-precision running sum.
 *
 * Layout: every matrix is row-major with a leading dimension in ELEMENTS
 * (A is M x K with lda >= K, B is K x N with ldb >= N, C is M x N with ldc >= N).
 * BF16 and FP16 operands arrive as their raw 16-bit patterns and are widened
 * exactly (a BF16 value is the top half of the FP32 with the same sign,
 * exponent and first 7 mantissa bits; an IEEE half is sign, 5-bit exponent
 * with bias 15, 10-bit mantissa, with subnormals at exponent 0).  FP8
 * operands (the OCP 8-bit formats) arrive as bytes: E4M3 is sign, 4-bit
 * exponent with bias 7, 3-bit mantissa, no infinities, S.1111.111 the only
 * NaN (largest finite 448); E5M2 is sign, 5-bit exponent with bias 15, 2-bit
 * mantissa, IEEE-style infinities and NaNs; both have subnormals at exponent
 * 0.  Every product of two such values is exact in double as well.
 *
 * Besides C, every entry point can also return D[i][j] = sum_k |A[i][k]|*|B[k][j]|,
 * the scale against which an error in C[i][j] is measured (max |dC| / D).
 *
 * Loop orders: the main routine runs i-k-j with a per-row accumulator and an
 * OpenMP loop over rows.  A second, independent j-i-k routine exists only so the
 * tests can brute-force one loop order against the other at tiny sizes.
 *
 * Fused epilogue (oracle_epilogue): section 13.10 of the same page names epilogue
 * fusion -- bias, activation, residual add or a type cast applied to the
 * accumulator before it is stored.  The reading taken here, written out in
 * fp64 on the exact product: y = act(alpha * acc + beta * c_old + bias[j]),
 * where c_old is the C already in memory (the residual, in the output type),
 * bias is one FP32 value per column, and act is none, ReLU (max(x, 0)) or
 * GELU (x times the standard normal CDF, Phi(x) = (1 + erf(x / sqrt 2)) / 2).
 * The result is returned unrounded; the cast to the output type is left to
 * the comparison, which allows for it.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (no -march flags, so
 * x86 and Arm hosts give the same bits).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double widen_bf16(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double widen_f16(uint16_t bits)
{
    const int sign = bits >> 15, e = (bits >> 10) & 31, m = bits & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);     /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

static double widen_e4m3(uint8_t bits)
{
    const int sign = bits >> 7, e = (bits >> 3) & 15, m = bits & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);                  /* subnormal: (m/8) * 2^-6 */
    else
        v = ldexp((double)(8 + m), e - 10);        /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

static double widen_e5m2(uint8_t bits)
{
    const int sign = bits >> 7, e = (bits >> 2) & 31, m = bits & 3;
    double v;
    if (e == 31)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)m, -16);                 /* subnormal: (m/4) * 2^-14 */
    else
        v = ldexp((double)(4 + m), e - 17);        /* (1 + m/4) * 2^(e-15) */
    return sign ? -v : v;
}

/* The 256 values of an 8-bit format. */
enum { FMT8_E4M3 = 0, FMT8_E5M2 = 1 };

static void fill_table8(int fmt, double *tab)
{
    for (int b = 0; b < 256; ++b)
        tab[b] = fmt == FMT8_E5M2 ? widen_e5m2((uint8_t)b) : widen_e4m3((uint8_t)b);
}

/* 16-bit operand formats */
enum { FMT_BF16 = 0, FMT_F16 = 1 };

static double widen16(uint16_t bits, int fmt) { return fmt == FMT_F16 ? widen_f16(bits) : widen_bf16(bits); }

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One output row i of C (and optionally of D), k ascending, fp64 sums.
 * a_at(k) and b_row(k) are expressed by the two element types below. */
static void row_f32(int64_t i, int64_t N, int64_t K, const float *A, int64_t lda,
                    const float *B, int64_t ldb, double *c, double *d)
{
    for (int64_t j = 0; j < N; ++j) c[j] = 0.0;
    if (d) for (int64_t j = 0; j < N; ++j) d[j] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double a = (double)A[i * lda + k];
        const float *b = B + k * ldb;
        for (int64_t j = 0; j < N; ++j) c[j] += a * (double)b[j];
        if (d) {
            const double aa = fabs(a);
            for (int64_t j = 0; j < N; ++j) d[j] += aa * fabs((double)b[j]);
        }
    }
}

static void row_h16(int fmt, int64_t i, int64_t N, int64_t K, const uint16_t *A, int64_t lda,
                    const uint16_t *B, int64_t ldb, double *c, double *d, double *bw)
{
    for (int64_t j = 0; j < N; ++j) c[j] = 0.0;
    if (d) for (int64_t j = 0; j < N; ++j) d[j] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double a = widen16(A[i * lda + k], fmt);
        const uint16_t *b = B + k * ldb;
        if (fmt == FMT_F16)
            for (int64_t j = 0; j < N; ++j) bw[j] = widen_f16(b[j]);
        else
            for (int64_t j = 0; j < N; ++j) bw[j] = widen_bf16(b[j]);
        for (int64_t j = 0; j < N; ++j) c[j] += a * bw[j];
        if (d) {
            const double aa = fabs(a);
            for (int64_t j = 0; j < N; ++j) d[j] += aa * fabs(bw[j]);
        }
    }
}

static void row_u8(const double *tab, int64_t i, int64_t N, int64_t K, const uint8_t *A, int64_t lda,
                   const uint8_t *B, int64_t ldb, double *c, double *d, double *bw)
{
    for (int64_t j = 0; j < N; ++j) c[j] = 0.0;
    if (d) for (int64_t j = 0; j < N; ++j) d[j] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double a = tab[A[i * lda + k]];
        const uint8_t *b = B + k * ldb;
        for (int64_t j = 0; j < N; ++j) bw[j] = tab[b[j]];
        for (int64_t j = 0; j < N; ++j) c[j] += a * bw[j];
        if (d) {
            const double aa = fabs(a);
            for (int64_t j = 0; j < N; ++j) d[j] += aa * fabs(bw[j]);
        }
    }
}

/* Full C (M x N, leading dimension ldc) and optional D (leading dimension ldd). */
void oracle_gemm_f32(int64_t M, int64_t N, int64_t K,
                     const float *A, int64_t lda, const float *B, int64_t ldb,
                     double *C, int64_t ldc, double *D, int64_t ldd)
{
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i)
        row_f32(i, N, K, A, lda, B, ldb, C + i * ldc, D ? D + i * ldd : NULL);
}

static void gemm_h16(int fmt, int64_t M, int64_t N, int64_t K,
                     const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                     double *C, int64_t ldc, double *D, int64_t ldd)
{
    #pragma omp parallel
    {
        double *bw = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        #pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < M; ++i)
            row_h16(fmt, i, N, K, A, lda, B, ldb, C + i * ldc, D ? D + i * ldd : NULL, bw);
        free(bw);
    }
}

void oracle_gemm_bf16(int64_t M, int64_t N, int64_t K,
                      const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                      double *C, int64_t ldc, double *D, int64_t ldd)
{
    gemm_h16(FMT_BF16, M, N, K, A, lda, B, ldb, C, ldc, D, ldd);
}

void oracle_gemm_f16(int64_t M, int64_t N, int64_t K,
                     const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                     double *C, int64_t ldc, double *D, int64_t ldd)
{
    gemm_h16(FMT_F16, M, N, K, A, lda, B, ldb, C, ldc, D, ldd);
}

/* Only the rows listed in rows[0..nrows): C and D are dense nrows x N outputs.
 * Used to check full-size problems where the whole product would take too long. */
void oracle_gemm_rows_f32(int64_t M, int64_t N, int64_t K,
                          const float *A, int64_t lda, const float *B, int64_t ldb,
                          const int64_t *rows, int64_t nrows, double *C, double *D)
{
    (void)M;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r)
        row_f32(rows[r], N, K, A, lda, B, ldb, C + r * N, D ? D + r * N : NULL);
}

static void rows_h16(int fmt, int64_t N, int64_t K, const uint16_t *A, int64_t lda, const uint16_t *B,
                     int64_t ldb, const int64_t *rows, int64_t nrows, double *C, double *D)
{
    #pragma omp parallel
    {
        double *bw = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        #pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r)
            row_h16(fmt, rows[r], N, K, A, lda, B, ldb, C + r * N, D ? D + r * N : NULL, bw);
        free(bw);
    }
}

void oracle_gemm_rows_bf16(int64_t M, int64_t N, int64_t K,
                           const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                           const int64_t *rows, int64_t nrows, double *C, double *D)
{
    (void)M;
    rows_h16(FMT_BF16, N, K, A, lda, B, ldb, rows, nrows, C, D);
}

void oracle_gemm_rows_f16(int64_t M, int64_t N, int64_t K,
                          const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                          const int64_t *rows, int64_t nrows, double *C, double *D)
{
    (void)M;
    rows_h16(FMT_F16, N, K, A, lda, B, ldb, rows, nrows, C, D);
}

static void gemm_u8(int fmt, int64_t M, int64_t N, int64_t K, const uint8_t *A, int64_t lda, const uint8_t *B,
                    int64_t ldb, double *C, int64_t ldc, double *D, int64_t ldd)
{
    double tab[256];
    fill_table8(fmt, tab);
    #pragma omp parallel
    {
        double *bw = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        #pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < M; ++i)
            row_u8(tab, i, N, K, A, lda, B, ldb, C + i * ldc, D ? D + i * ldd : NULL, bw);
        free(bw);
    }
}

void oracle_gemm_e4m3(int64_t M, int64_t N, int64_t K, const uint8_t *A, int64_t lda, const uint8_t *B, int64_t ldb,
                      double *C, int64_t ldc, double *D, int64_t ldd)
{
    gemm_u8(FMT8_E4M3, M, N, K, A, lda, B, ldb, C, ldc, D, ldd);
}

void oracle_gemm_e5m2(int64_t M, int64_t N, int64_t K, const uint8_t *A, int64_t lda, const uint8_t *B, int64_t ldb,
                      double *C, int64_t ldc, double *D, int64_t ldd)
{
    gemm_u8(FMT8_E5M2, M, N, K, A, lda, B, ldb, C, ldc, D, ldd);
}

static void rows_u8(int fmt, int64_t N, int64_t K, const uint8_t *A, int64_t lda, const uint8_t *B, int64_t ldb,
                    const int64_t *rows, int64_t nrows, double *C, double *D)
{
    double tab[256];
    fill_table8(fmt, tab);
    #pragma omp parallel
    {
        double *bw = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        #pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r)
            row_u8(tab, rows[r], N, K, A, lda, B, ldb, C + r * N, D ? D + r * N : NULL, bw);
        free(bw);
    }
}

void oracle_gemm_rows_e4m3(int64_t M, int64_t N, int64_t K, const uint8_t *A, int64_t lda, const uint8_t *B,
                           int64_t ldb, const int64_t *rows, int64_t nrows, double *C, double *D)
{
    (void)M;
    rows_u8(FMT8_E4M3, N, K, A, lda, B, ldb, rows, nrows, C, D);
}

void oracle_gemm_rows_e5m2(int64_t M, int64_t N, int64_t K, const uint8_t *A, int64_t lda, const uint8_t *B,
                           int64_t ldb, const int64_t *rows, int64_t nrows, double *C, double *D)
{
    (void)M;
    rows_u8(FMT8_E5M2, N, K, A, lda, B, ldb, rows, nrows, C, D);
}

/* Second loop order (j outer, then i, then k), single-threaded, for brute-force
 * self-checks of the routine above on tiny sizes. */
void oracle_gemm_f32_jik(int64_t M, int64_t N, int64_t K,
                         const float *A, int64_t lda, const float *B, int64_t ldb,
                         double *C, int64_t ldc)
{
    for (int64_t j = 0; j < N; ++j)
        for (int64_t i = 0; i < M; ++i) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k)
                s += (double)A[i * lda + k] * (double)B[k * ldb + j];
            C[i * ldc + j] = s;
        }
}

static void jik_h16(int fmt, int64_t M, int64_t N, int64_t K, const uint16_t *A, int64_t lda, const uint16_t *B,
                    int64_t ldb, double *C, int64_t ldc)
{
    for (int64_t j = 0; j < N; ++j)
        for (int64_t i = 0; i < M; ++i) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k)
                s += widen16(A[i * lda + k], fmt) * widen16(B[k * ldb + j], fmt);
            C[i * ldc + j] = s;
        }
}

void oracle_gemm_bf16_jik(int64_t M, int64_t N, int64_t K,
                          const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                          double *C, int64_t ldc)
{
    jik_h16(FMT_BF16, M, N, K, A, lda, B, ldb, C, ldc);
}

void oracle_gemm_f16_jik(int64_t M, int64_t N, int64_t K,
                         const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                         double *C, int64_t ldc)
{
    jik_h16(FMT_F16, M, N, K, A, lda, B, ldb, C, ldc);
}

static void jik_u8(int fmt, int64_t M, int64_t N, int64_t K, const uint8_t *A, int64_t lda, const uint8_t *B,
                   int64_t ldb, double *C, int64_t ldc)
{
    for (int64_t j = 0; j < N; ++j)
        for (int64_t i = 0; i < M; ++i) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const uint8_t a = A[i * lda + k], b = B[k * ldb + j];
                s += fmt == FMT8_E5M2 ? widen_e5m2(a) * widen_e5m2(b) : widen_e4m3(a) * widen_e4m3(b);
            }
            C[i * ldc + j] = s;
        }
}

void oracle_gemm_e4m3_jik(int64_t M, int64_t N, int64_t K, const uint8_t *A, int64_t lda, const uint8_t *B,
                          int64_t ldb, double *C, int64_t ldc)
{
    jik_u8(FMT8_E4M3, M, N, K, A, lda, B, ldb, C, ldc);
}

void oracle_gemm_e5m2_jik(int64_t M, int64_t N, int64_t K, const uint8_t *A, int64_t lda, const uint8_t *B,
                          int64_t ldb, double *C, int64_t ldc)
{
    jik_u8(FMT8_E5M2, M, N, K, A, lda, B, ldb, C, ldc);
}

/* Exact widening of n BF16 / FP16 patterns, exposed so the tests can pin it. */
void oracle_widen_bf16(const uint16_t *src, double *dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = widen_bf16(src[i]);
}

void oracle_widen_f16(const uint16_t *src, double *dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = widen_f16(src[i]);
}

/* ... and of n FP8 bytes (the j-i-k routines call these directly, not the table). */
void oracle_widen_e4m3(const uint8_t *src, double *dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = widen_e4m3(src[i]);
}

void oracle_widen_e5m2(const uint8_t *src, double *dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = widen_e5m2(src[i]);
}

/* ------------------------------------------------------------ epilogue --- */
enum { ACT_NONE = 0, ACT_RELU = 1, ACT_GELU = 2 };
enum { OUT_F32 = 0, OUT_BF16 = 1, OUT_F16 = 2 };

static double read_old(const void *c_old, int out, int64_t idx)
{
    if (out == OUT_BF16) return widen_bf16(((const uint16_t *)c_old)[idx]);
    if (out == OUT_F16) return widen_f16(((const uint16_t *)c_old)[idx]);
    return (double)((const float *)c_old)[idx];
}

/* Y[i][j] = act(alpha * acc[i][j] + beta * c_old[i][j] + bias[j]) for an M x N
 * block.  c_old (element type `out`) is read only when beta != 0; bias may be
 * NULL.  acc, c_old and Y have their own leading dimensions. */
void oracle_epilogue(int64_t M, int64_t N, const double *acc, int64_t ld_acc, double alpha, double beta,
                     const void *c_old, int out, int64_t ld_old, const float *bias, int act,
                     double *Y, int64_t ldy)
{
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double x = alpha * acc[i * ld_acc + j];
            if (beta != 0.0) x += beta * read_old(c_old, out, i * ld_old + j);
            if (bias) x += (double)bias[j];
            if (act == ACT_RELU)
                x = x > 0.0 ? x : 0.0;
            else if (act == ACT_GELU)
                x = x * 0.5 * (1.0 + erf(x / sqrt(2.0)));
            Y[i * ldy + j] = x;
        }
}
