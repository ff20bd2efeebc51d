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

/* ------------------------------------------------------ MXFP8 quantisation */

/*
 * Round an fp64 value to the nearest E4M3 ("e4m3fn") code, ties to even.
 * E4M3 keeps 4 significant bits; the smallest normal exponent is -6 and
 * below it the spacing is 2^-9; the largest finite value is 448.  Values
 * of magnitude above 448 are outside the encoder's domain here (the
 * quantiser below never produces them).
 */
uint8_t oracle_f64_to_e4m3_rne(double v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (isnan(v))
        return (uint8_t)(sign | 0x7F);
    if (a == 0.0)
        return sign;
    int ex;
    (void)frexp(a, &ex);
    int lead = ex - 1;                        /* exponent of the leading bit */
    if (lead < -6)
        lead = -6;
    double quantum = ldexp(1.0, lead - 3);
    double r = rint(a / quantum) * quantum;   /* ties to even */
    if (r == 0.0)
        return sign;
    /* encode r: normal if r >= 2^-6, else subnormal (exponent field 0) */
    if (r < ldexp(1.0, -6))
        return (uint8_t)(sign | (uint8_t)(r / ldexp(1.0, -9)));
    int e2;
    double m = frexp(r, &e2);                 /* r = m * 2^e2, m in [0.5, 1) */
    int biased = (e2 - 1) + 7;
    int mant = (int)((m * 2.0 - 1.0) * 8.0);  /* exact: r has 4 significant bits */
    return (uint8_t)(sign | (biased << 3) | mant);
}

/*
 * MXFP8 quantisation of float rows X [rows, K] (pitch ldx elements): for each
 * block of 32 consecutive k (the last block may be partial), amax = the
 * largest |x| over the block's finite values, the scale exponent e is the
 * smallest integer with amax <= 448 * 2^e (clamped to [-127, 127]; amax = 0
 * gives e = -127), SF[r, b] = e + 127 (UE8M0) and Q[r, k] = RNE-to-E4M3 of
 * x * 2^-e; a NaN or infinite x encodes as E4M3 NaN with its sign.
 */
void oracle_mxfp8_quantize(const float *X, int64_t rows, int64_t K, int64_t ldx,
                           uint8_t *Q, int64_t ldq, uint8_t *SF, int64_t ldsf)
{
    int64_t nblk = (K + 31) / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nblk; ++b) {
            int64_t k0 = b * 32, k1 = k0 + 32 < K ? k0 + 32 : K;
            double amax = 0.0;
            for (int64_t k = k0; k < k1; ++k) {
                double x = (double)X[r * ldx + k];
                if (isfinite(x) && fabs(x) > amax)
                    amax = fabs(x);
            }
            int e = -127;
            if (amax > 0.0) {
                /* exact search: start at the float guess, then step to the minimum */
                e = (int)ceil(log2(amax / 448.0));
                while (amax > ldexp(448.0, e))
                    ++e;
                while (e > -127 && amax <= ldexp(448.0, e - 1))
                    --e;
                if (e > 127)
                    e = 127;
                if (e < -127)
                    e = -127;
            }
            SF[r * ldsf + b] = (uint8_t)(e + 127);
            for (int64_t k = k0; k < k1; ++k) {
                double x = (double)X[r * ldx + k];
                if (!isfinite(x))
                    Q[r * ldq + k] = (uint8_t)((signbit(x) ? 0x80 : 0x00) | 0x7F);
                else
                    Q[r * ldq + k] = oracle_f64_to_e4m3_rne(ldexp(x, -e));
            }
        }
    }
}

/* --------------------------------------------------------- fused epilogue */

/*
 * The epilogue fused into the TMEM -> register readback (b200-tmem-
 * lifecycle-planner, "A1 -- Case 1: dense MMA accumulator": the warpgroup
 * reads the fp32 accumulator back into registers for the cast/epilogue/store;
 * b200-gemm-optimization-ladder, "B -- Boundaries", "Do not use when": custom
 * fusion is a reason to own the kernel).  The pages name no particular
 * epilogue; this is the plain linear-layer one.  Given the exact sums P of
 * one of the GEMMs above, in fp64:
 *
 *     v[i][j] = alpha * P[i][j] + beta * C[i][j] + bias[j]
 *     D[i][j] = act(v[i][j])
 *
 *   act 0: identity.
 *   act 1: ReLU, 0 where v < 0 and v otherwise (NaN stays NaN).
 *   act 2: GELU, v * Phi(v) with Phi the standard normal distribution
 *          function, Phi(v) = (1 + erf(v / sqrt 2)) / 2.
 *
 * C (decoded, [M,N] with pitch ldc) and bias (decoded, [N]) may be NULL, in
 * which case their term is absent.  out is dense [M,N].
 */
static double act_f64(double v, int act)
{
    if (act == 1) return v < 0.0 ? 0.0 : v;
    if (act == 2) return v * 0.5 * (1.0 + erf(v / sqrt(2.0)));
    return v;
}

void oracle_epilogue(const double *P, int64_t M, int64_t N, double alpha, double beta,
                     const double *C, int64_t ldc, const double *bias, int act, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double v = alpha * P[i * N + j];
            if (C) v += beta * C[i * ldc + j];
            if (bias) v += bias[j];
            out[i * N + j] = act_f64(v, act);
        }
}
