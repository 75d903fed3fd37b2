/*
 * oracle.c -- plain, slow fp64 reference for the dense GEMM C = A * B^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library.
 *
 * What it computes (the plain definition the pages build every kernel from):
 *   "Matrix Multiplication on NVIDIA's Blackwell", background section on the
 *   definition of matmul (the triple loop over row, col, inner), and the
 *   naive "Kernel 1" listing, which indexes b[col, k]: B is stored N x K,
 *   K-major ("B is K x N, already transposed", optimisation roadmap section).
 *
 *     C[i][j] = round_dtype( sum_{k=0}^{K-1} A[i][k] * B[j][k] )
 *
 *   - every bf16 / fp16 input is widened exactly to double;
 *   - products are exact in double (8x8 or 11x11 significand bits) and are
 *     summed in double in plain order k = 0 .. K-1;
 *   - the double sum is rounded once, directly, to the output format with
 *     IEEE-754 round-to-nearest-even (the pages do not state the rounding;
 *     this is the reading taken), overflow to +-inf.
 *
 * The two 16-bit formats are decoded and encoded here from their definitions
 * (sign | exponent | significand, with subnormals):
 *   bf16: 1 + 8 + 7 bits, bias 127 (the "BF16 data type" figure of the
 *         Blackwell deep dive, Kernel 1 section);
 *   fp16: 1 + 5 + 10 bits, bias 15 (IEEE-754 binary16; the CuTeDSL post
 *         times fp16 tensors, "how I measured" section).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_BF16 0
#define ORACLE_FP16 1

typedef struct {
    int mant_bits; /* explicit significand bits          */
    int exp_bits;  /* exponent field width               */
    int bias;      /* exponent bias                       */
} fmt16_t;

static const fmt16_t k_formats[2] = {
    {7, 8, 127}, /* bf16 */
    {10, 5, 15}, /* fp16 */
};

static int valid_dtype(int dtype) { return dtype == ORACLE_BF16 || dtype == ORACLE_FP16; }

/* Exact value of a 16-bit pattern as a double. */
double oracle_decode(uint16_t bits, int dtype)
{
    const fmt16_t f = k_formats[dtype ? 1 : 0];
    const int exp_all = (1 << f.exp_bits) - 1;
    const int sign = (bits >> 15) & 1;
    const int e = (bits >> f.mant_bits) & exp_all;
    const int m = bits & ((1 << f.mant_bits) - 1);
    double v;
    if (e == exp_all)
        v = m ? NAN : INFINITY;
    else if (e == 0) /* subnormal: m * 2^(emin - mant_bits), emin = 1 - bias */
        v = ldexp((double)m, 1 - f.bias - f.mant_bits);
    else /* normal: (2^mant_bits + m) * 2^(e - bias - mant_bits) */
        v = ldexp((double)(m | (1 << f.mant_bits)), e - f.bias - f.mant_bits);
    return sign ? -v : v;
}

/* Round a double to the nearest representable 16-bit value, ties to the
 * value whose significand is even; returns the bit pattern. */
uint16_t oracle_round(double x, int dtype)
{
    const fmt16_t f = k_formats[dtype ? 1 : 0];
    const uint16_t exp_all = (uint16_t)((1 << f.exp_bits) - 1);
    const uint16_t inf_bits = (uint16_t)(exp_all << f.mant_bits);
    const uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x))
        return (uint16_t)(sign | inf_bits | (1u << (f.mant_bits - 1))); /* quiet NaN */
    const double a = fabs(x);
    if (isinf(a))
        return (uint16_t)(sign | inf_bits);
    if (a == 0.0)
        return sign;

    const int emin = 1 - f.bias; /* exponent of the smallest normal   */
    const int emax = f.bias;     /* exponent of the largest binade    */
    int e2;
    (void)frexp(a, &e2); /* a = frac * 2^e2, frac in [0.5, 1)  */
    int E = e2 - 1;      /* a = 1.xxx * 2^E                     */
    if (E < emin)
        E = emin; /* subnormal range: fixed spacing      */
    if (E > emax)
        return (uint16_t)(sign | inf_bits);

    /* Spacing of representable values in the binade of E. a / q is exact:
     * q is a power of two and the quotient stays far inside double range. */
    const double q = ldexp(1.0, E - f.mant_bits);
    const double n = a / q; /* < 2^(mant_bits + 1)                */
    const double fl = floor(n);
    const double rem = n - fl;
    double r = fl;
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0))
        r = fl + 1.0;

    const uint32_t hidden = 1u << f.mant_bits;
    uint32_t ri = (uint32_t)r;
    if (ri >= (hidden << 1)) { /* rounded up into the next binade   */
        ri = hidden;
        E += 1;
        if (E > emax)
            return (uint16_t)(sign | inf_bits);
    }
    if (ri < hidden) /* subnormal (E == emin) */
        return (uint16_t)(sign | ri);
    return (uint16_t)(sign | (uint16_t)((E + f.bias) << f.mant_bits) | (uint16_t)(ri - hidden));
}

/* Element-wise helpers for the Python side. */
void oracle_decode_array(const uint16_t *bits, double *out, int64_t n, int dtype)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_decode(bits[i], dtype);
}

void oracle_round_array(const double *x, uint16_t *out, int64_t n, int dtype)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_round(x[i], dtype);
}

/* Widening table: value of every 16-bit pattern, filled from oracle_decode
 * once per format before a product loop (a lookup, not a different rule). */
static double k_widen[2][65536];
static int k_widen_ready[2];

static void fill_widen_table(int dtype)
{
    if (k_widen_ready[dtype])
        return;
    for (int b = 0; b < 65536; ++b)
        k_widen[dtype][b] = oracle_decode((uint16_t)b, dtype);
    k_widen_ready[dtype] = 1;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * C_sub = rows x cols block of round(A * B^T).
 *
 *   A    : M x K bit patterns, row stride lda (elements), lda >= K
 *   B    : N x K bit patterns, row stride ldb (elements), ldb >= K
 *   rows : nrows row indices of C to compute (NULL: all M rows, nrows = M)
 *   cols : ncols column indices of C to compute (NULL: all N cols, ncols = N)
 *   Cout : nrows x ncols dense output bit patterns (may be NULL)
 *   Cacc : nrows x ncols dense unrounded double sums (may be NULL)
 *   nthreads : OpenMP threads (<= 0: the runtime default)
 *
 * Returns 0, or -1 on a bad argument.
 */
int oracle_gemm(const uint16_t *A, const uint16_t *B, uint16_t *Cout, double *Cacc,
                int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int dtype,
                const int64_t *rows, int64_t nrows, const int64_t *cols, int64_t ncols,
                int nthreads)
{
    if (!valid_dtype(dtype) || M < 0 || N < 0 || K < 0 || lda < K || ldb < K)
        return -1;
    if (!rows)
        nrows = M;
    if (!cols)
        ncols = N;
    if (nrows < 0 || ncols < 0)
        return -1;
    if (K > 0 && ((M > 0 && !A) || (N > 0 && !B)))
        return -1;
    for (int64_t r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M)
            return -1;
    for (int64_t c = 0; cols && c < ncols; ++c)
        if (cols[c] < 0 || cols[c] >= N)
            return -1;
    if (nrows == 0 || ncols == 0)
        return 0;

#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#else
    (void)nthreads;
#endif
    int err = 0;
    fill_widen_table(dtype); /* before the threads start */
    const double *widen = k_widen[dtype];

#pragma omp parallel num_threads(nthreads)
    {
        /* the current row of A, widened to double */
        double *arow = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        if (!arow) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!arow)
                continue;
            const int64_t i = rows ? rows[r] : r;
            for (int64_t k = 0; k < K; ++k)
                arow[k] = widen[A[i * lda + k]];
            for (int64_t c = 0; c < ncols; ++c) {
                const int64_t j = cols ? cols[c] : c;
                const uint16_t *brow = B + j * ldb;
                double s = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    s += arow[k] * widen[brow[k]];
                if (Cacc)
                    Cacc[r * ncols + c] = s;
                if (Cout)
                    Cout[r * ncols + c] = oracle_round(s, dtype);
            }
        }
        free(arow);
    }
    return err ? -1 : 0;
}
