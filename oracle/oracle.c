/*
 * Reference GEMM oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU statement of what the tcgen05 GEMM
 * computes, in IEEE fp64.  Only the test-suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this library; the product path never
 * does, and this file shares no header, helper or table with the CUDA code.
 *
 * What is computed (b200-gemm-optimization-ladder, "A1 -- The nine-level
 * route": every level keeps the data path GMEM->SMEM->tcgen05->TMEM->
 * registers/SMEM->GMEM and only changes scheduling; "E -- Executable steps",
 * step 1 "baseline contract": math definition, layout, dtype):
 *
 *     D[i][j] = sum_{k<K} a(i,k) * b(j,k)
 *
 * with A stored [M,K] row-major (leading dimension lda elements) and B stored
 * [N,K] K-major (leading dimension ldb elements), i.e. D = A * B^T.
 *
 *   bf16 variant : a(i,k) = bf16(A[i*lda+k]),  b(j,k) = bf16(B[j*ldb+k]).
 *   MXFP8 variant: a(i,k) = 2^(SFA[i*ldsfa + k/32] - 127) * e4m3(A[i*lda+k]),
 *                  b(j,k) = 2^(SFB[j*ldsfb + k/32] - 127) * e4m3(B[j*ldb+k])
 *     (block-scaled operands whose scale factors are staged through TMEM:
 *      b200-tmem-lifecycle-planner, "A1 -- Case 2: block-scaled MMA").
 *
 * The device accumulates in fp32 in TMEM (b200-tmem-lifecycle-planner, "A1 --
 * Case 1: dense MMA accumulator"); the oracle accumulates the same products in
 * fp64 in natural k order, with no blocking or reordering, and also returns
 * S[i][j] = sum_k |a(i,k) * b(j,k)|, the scale of the rounding-error bound.
 *
 * Number formats, written from their definitions:
 *   bf16  : the upper 16 bits of an IEEE binary32.
 *   E4M3  : OCP FP8 "E4M3FN": 1 sign, 4 exponent (bias 7), 3 mantissa bits;
 *           exponent field 0 is subnormal (m * 2^-9); S.1111.111 is NaN;
 *           no infinities; largest finite value 448.
 *   UE8M0 : unsigned 8-bit exponent e meaning 2^(e-127); e = 255 is NaN.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- decoders */

double oracle_bf16_to_f64(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oracle_e4m3_to_f64(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);                    /* subnormal: m/8 * 2^(1-7) */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);     /* normal */
    return sign ? -v : v;
}

double oracle_ue8m0_to_f64(uint8_t e)
{
    if (e == 0xFF)
        return NAN;
    return ldexp(1.0, (int)e - 127);
}

/*
 * Round an fp64 value to bfloat16, round-to-nearest-even, and return the bit
 * pattern.  bf16 keeps 8 significant bits; its smallest normal exponent is
 * -126 and below that the spacing is fixed at 2^-133.  The rounded value is
 * always representable in binary32, so the bits are read off a float.
 */
uint16_t oracle_f64_to_bf16_rne(double x)
{
    if (isnan(x))
        return 0x7FC0;
    if (x == 0.0 || isinf(x)) {
        float f = (float)x;
        uint32_t u;
        memcpy(&u, &f, sizeof u);
        return (uint16_t)(u >> 16);
    }
    int ex;
    (void)frexp(x, &ex);           /* |x| = f * 2^ex, f in [0.5, 1) */
    int lead = ex - 1;             /* exponent of the leading bit */
    if (lead < -126)
        lead = -126;
    double quantum = ldexp(1.0, lead - 7);
    double r = rint(x / quantum) * quantum;   /* rint: ties to even */
    if (fabs(r) >= ldexp(1.0, 128))
        r = x > 0 ? INFINITY : -INFINITY;
    float f = (float)r;            /* exact: r is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------- GEMMs */

/* One output element: the plain inner product over k in natural order. */
static void dot_bf16(const uint16_t *a, const uint16_t *b, int64_t K,
                     double *d, double *s)
{
    double acc = 0.0, abs_acc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double p = oracle_bf16_to_f64(a[k]) * oracle_bf16_to_f64(b[k]);
        acc += p;
        abs_acc += fabs(p);
    }
    *d = acc;
    *s = abs_acc;
}

/* Full D = A * B^T for bf16 operands.  D and S are dense [M,N] fp64. */
void oracle_gemm_bf16(const uint16_t *A, const uint16_t *B,
                      int64_t M, int64_t N, int64_t K,
                      int64_t lda, int64_t ldb, double *D, double *S)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j)
            dot_bf16(A + i * lda, B + j * ldb, K, &D[i * N + j], &S[i * N + j]);
}

/* Selected entries (rows[t], cols[t]) of D = A * B^T, for sizes where the
 * full product is too slow on a CPU. */
void oracle_gemm_bf16_entries(const uint16_t *A, const uint16_t *B,
                              int64_t K, int64_t lda, int64_t ldb,
                              const int64_t *rows, const int64_t *cols,
                              int64_t n, double *D, double *S)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t)
        dot_bf16(A + rows[t] * lda, B + cols[t] * ldb, K, &D[t], &S[t]);
}

static void dot_mxfp8(const uint8_t *a, const uint8_t *b,
                      const uint8_t *sfa, const uint8_t *sfb, int64_t K,
                      double *d, double *s)
{
    double acc = 0.0, abs_acc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double av = oracle_ue8m0_to_f64(sfa[k / 32]) * oracle_e4m3_to_f64(a[k]);
        double bv = oracle_ue8m0_to_f64(sfb[k / 32]) * oracle_e4m3_to_f64(b[k]);
        double p = av * bv;
        acc += p;
        abs_acc += fabs(p);
    }
    *d = acc;
    *s = abs_acc;
}

/* Full D = A * B^T for block-scaled E4M3 operands with one UE8M0 scale per
 * 32 consecutive k.  SFA is [M, ldsfa] row-major, SFB is [N, ldsfb]. */
void oracle_gemm_mxfp8(const uint8_t *A, const uint8_t *B,
                       const uint8_t *SFA, const uint8_t *SFB,
                       int64_t M, int64_t N, int64_t K,
                       int64_t lda, int64_t ldb, int64_t ldsfa, int64_t ldsfb,
                       double *D, double *S)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j)
            dot_mxfp8(A + i * lda, B + j * ldb, SFA + i * ldsfa, SFB + j * ldsfb,
                      K, &D[i * N + j], &S[i * N + j]);
}

void oracle_gemm_mxfp8_entries(const uint8_t *A, const uint8_t *B,
                               const uint8_t *SFA, const uint8_t *SFB,
                               int64_t K, int64_t lda, int64_t ldb,
                               int64_t ldsfa, int64_t ldsfb,
                               const int64_t *rows, const int64_t *cols,
                               int64_t n, double *D, double *S)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t)
        dot_mxfp8(A + rows[t] * lda, B + cols[t] * ldb,
                  SFA + rows[t] * ldsfa, SFB + cols[t] * ldsfb, K, &D[t], &S[t]);
}

/* ------------------------------------------------ element-wise array forms */

void oracle_bf16_to_f64_array(const uint16_t *in, int64_t n, double *out)
{
    for (int64_t t = 0; t < n; ++t)
        out[t] = oracle_bf16_to_f64(in[t]);
}

void oracle_e4m3_to_f64_array(const uint8_t *in, int64_t n, double *out)
{
    for (int64_t t = 0; t < n; ++t)
        out[t] = oracle_e4m3_to_f64(in[t]);
}

void oracle_ue8m0_to_f64_array(const uint8_t *in, int64_t n, double *out)
{
    for (int64_t t = 0; t < n; ++t)
        out[t] = oracle_ue8m0_to_f64(in[t]);
}

void oracle_f64_to_bf16_rne_array(const double *in, int64_t n, uint16_t *out)
{
    for (int64_t t = 0; t < n; ++t)
        out[t] = oracle_f64_to_bf16_rne(in[t]);
}
