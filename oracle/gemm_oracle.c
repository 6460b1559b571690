/*
 * CPU oracle for the bf16 GEMM  D = A * B^T   -- TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference
 * arm may load this library.  The product path (the CUDA library under
 * warp_specialized_tma_gb300/) never links, loads or calls it, and the two share
 * no code, headers or constants.
 *
 * What it computes is the plain definition of the operation that the warp-
 * specialised matmul computes:
 *
 *   Fuser issue #3941, "Allow separate sub-DAG for load and compute warp groups
 *   with warp-specialized circular buffering", Pseudo-code: the compute warp
 *   group accumulates, over every cta-k step of an output tile, the products of
 *   the A and B operand tiles, and after the last step converts the fp32 sums to
 *   bf16 and stores them.  Both operands are read "K-major" (the contraction
 *   index is the contiguous one), so D[m][n] = sum_k A[m][k] * B[n][k].
 *
 * The oracle takes the same bf16 bit patterns as the GPU, widens them to fp64
 * (exact), forms every product in fp64 (exact: two 8-bit significands give at
 * most 16 bits), sums them in increasing k in one fp64 accumulator, and rounds
 * the fp64 sum ONCE to bf16, round-to-nearest, ties-to-even (IEEE 754
 * roundTiesToEven applied to the bf16 format: 1 sign bit, 8 exponent bits with
 * bias 127, 7 stored fraction bits).  No blocking, no reordering, no fusion.
 *
 * Parity status: pinned (see tests/test_oracle.py: exact brute force with
 * rationals, identity / permutation / all-ones closed forms, integer inputs,
 * an fp64 library matmul, hand-derived rounding cases, fp32->bf16 library
 * rounding).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> fp64.  A bf16 value is the top half of an IEEE binary32
 * pattern, so widening is a 16-bit shift into binary32 followed by an exact
 * binary32 -> binary64 conversion. */
double oracle_f64_from_bf16(uint16_t h)
{
    uint32_t w = (uint32_t)h << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* fp64 -> bf16, round to nearest, ties to even, from the definition.
 *
 * bf16 normal numbers are s * 2^E with E in [-126, 127] and an 8-bit significand
 * s in [128, 256) counted in units of 2^(E-7).  Below 2^-126 the grid is fixed
 * at 2^-133 (subnormals).  We scale |x| onto its grid (a power-of-two scaling,
 * exact in fp64), round the scaled value to an integer with ties to even, then
 * encode.  A carry to 256 moves to the next binade; past 2^127 * 255/128 the
 * result is infinity. */
uint16_t oracle_bf16_from_f64(double x)
{
    if (isnan(x))
        return (uint16_t)0x7FC0u;               /* one quiet NaN */
    uint16_t sign = signbit(x) ? (uint16_t)0x8000u : (uint16_t)0u;
    double ax = fabs(x);
    if (isinf(ax))
        return (uint16_t)(sign | 0x7F80u);
    if (ax == 0.0)
        return sign;

    int e;
    (void)frexp(ax, &e);          /* ax = f * 2^e, 0.5 <= f < 1 */
    int E = e - 1;                /* ax = 1.xxx * 2^E */
    int grid = (E >= -126) ? (E - 7) : -133;
    double q = ldexp(ax, -grid);  /* exact */
    double fl = floor(q);
    double rem = q - fl;          /* exact */
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0))
        fl += 1.0;

    uint32_t bits;
    if (grid == -133) {
        /* subnormal grid: fl in [0, 128]; 128 is exactly the smallest normal
         * 2^-126, whose encoding (exponent field 1, fraction 0) is 0x0080. */
        bits = (uint32_t)fl;
    } else {
        int Eb = E;
        if (fl == 256.0) {
            fl = 128.0;
            Eb += 1;
        }
        if (Eb > 127)
            return (uint16_t)(sign | 0x7F80u);
        bits = ((uint32_t)(Eb + 127) << 7) | ((uint32_t)fl - 128u);
    }
    return (uint16_t)(sign | bits);
}

/* Element-wise conversions over arrays (used by the tests' rounding pins). */
void oracle_bf16_from_f64_array(const double *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_from_f64(x[i]);
}

void oracle_f64_from_bf16_array(const uint16_t *h, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f64_from_bf16(h[i]);
}

/* D rows of  D = A * B^T.
 *
 *   A    : M x K bf16 patterns, row m at A + m*lda  (lda >= K)
 *   B    : N x K bf16 patterns, row n at B + n*ldb  (ldb >= K)
 *   rows : the m indices to compute (nrows of them); NULL means all M rows in
 *          order (nrows must then equal M)
 *   ref64, refbf16 : nrows x N outputs, row i at +i*N; either may be NULL
 *
 * Returns 0, or -1 on a bad argument (row index out of range, bad sizes). */
int oracle_gemm_rows(const uint16_t *A, int64_t lda,
                     const uint16_t *B, int64_t ldb,
                     int64_t M, int64_t N, int64_t K,
                     const int64_t *rows, int64_t nrows,
                     double *ref64, uint16_t *refbf16)
{
    if (M < 0 || N < 0 || K < 0 || nrows < 0 || lda < K || ldb < K)
        return -1;
    if (rows == NULL && nrows != M)
        return -1;
    if (rows != NULL)
        for (int64_t i = 0; i < nrows; ++i)
            if (rows[i] < 0 || rows[i] >= M)
                return -1;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        const uint16_t *a = A + m * lda;
        for (int64_t n = 0; n < N; ++n) {
            const uint16_t *b = B + n * ldb;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += oracle_f64_from_bf16(a[k]) * oracle_f64_from_bf16(b[k]);
            if (ref64)
                ref64[i * N + n] = acc;
            if (refbf16)
                refbf16[i * N + n] = oracle_bf16_from_f64(acc);
        }
    }
    return 0;
}

/* Rows of the fused form  D = alpha * (A * B^T) + beta * C + bias.
 *
 * The pages' epilogue (Fuser issue #3941, Pseudo-code: convert the fp32 sums
 * and store) is the place a GEMM fuses its element-wise tail; this is the
 * plain definition of that tail.  Every term is formed in fp64 from the same
 * inputs the GPU gets -- alpha and beta as given (fp32 values, exact in fp64),
 * C[m][n] and bias[n] widened from bf16 -- and the total is rounded ONCE to
 * bf16.  C (row pitch ldc) and bias may be NULL, meaning 0.  Outputs as in
 * oracle_gemm_rows (ref64 is the unrounded fp64 value).  Returns 0 or -1. */
int oracle_gemm_fused_rows(const uint16_t *A, int64_t lda,
                           const uint16_t *B, int64_t ldb,
                           int64_t M, int64_t N, int64_t K,
                           const int64_t *rows, int64_t nrows,
                           double alpha, double beta,
                           const uint16_t *C, int64_t ldc, const uint16_t *bias,
                           double *ref64, uint16_t *refbf16)
{
    if (M < 0 || N < 0 || K < 0 || nrows < 0 || lda < K || ldb < K || (C && ldc < N))
        return -1;
    if (rows == NULL && nrows != M)
        return -1;
    if (rows != NULL)
        for (int64_t i = 0; i < nrows; ++i)
            if (rows[i] < 0 || rows[i] >= M)
                return -1;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        const uint16_t *a = A + m * lda;
        for (int64_t n = 0; n < N; ++n) {
            const uint16_t *b = B + n * ldb;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += oracle_f64_from_bf16(a[k]) * oracle_f64_from_bf16(b[k]);
            double v = alpha * acc;
            if (C)
                v += beta * oracle_f64_from_bf16(C[m * ldc + n]);
            if (bias)
                v += oracle_f64_from_bf16(bias[n]);
            if (ref64)
                ref64[i * N + n] = v;
            if (refbf16)
                refbf16[i * N + n] = oracle_bf16_from_f64(v);
        }
    }
    return 0;
}

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
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
