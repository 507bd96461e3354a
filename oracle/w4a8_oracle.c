/*
 * w4a8_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow CPU statement of the W4A8 block-64 quantized linear.  It exists
 * so that the CUDA path can be checked against something written independently
 * of it.  Only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg load this file; the product library never links or calls it, and it shares
 * no code, header or table with the CUDA sources.
 *
 * Source of the method: "MNN LLM inference on the SpacemiT K3 (RVV, IME2, TCM)"
 * (zhaode.wang blog), section 3 ("asymmetric W4B64 expansion"):
 *   eq. (1)  w ~= s_w (q_w - z_w)                       HQQ block-64 asymmetric W4
 *   eq. (2)  sum_i a_i w_i ~= s_w (sum_i a_i q_i - z_w sum_i a_i)
 *   eq. (3)  a8 = 16 * (a8 >> 4) + (a8 & 0x0f)          high nibble signed, low unsigned
 * and section 4 (prefill): one pass does absmax -> scale -> packed INT8 A plus the
 * per-block input row sum ("srcKernelSum"); the epilogue applies scale, zero-point
 * correction and bias directly to the final output.
 *
 * Readings taken where the page is silent (each one is listed in the design notes):
 *   - activation scale s_a = absmax / 127 as an fp32 IEEE division, and the code is
 *     a_q = clamp(roundf(x / s_a), -127, 127) with an fp32 IEEE division and
 *     round-half-away-from-zero; a row whose s_a is 0 (an all-zero row, or absmax / 127
 *     underflowing to 0) gives a_q = 0;
 *   - one (s_w, z_w) fp16 pair per 64 consecutive K elements of one output row n;
 *     z_w is a real fp16 value, q is unsigned 0..15;
 *   - packed weights: byte wq[n][k/2] holds k even in its low nibble, k odd in
 *     its high nibble;
 *   - bias is optional fp32 [N]; the output is fp32 row-major [M][N]; no clamp.
 *
 * Arithmetic: integer stages in int32/int64, the output in fp64.  The fp16 inputs
 * are decoded by this file's own routine.  Build with -ffp-contract=off so that
 * no multiply-add is fused behind the reader's back.
 */
#include <stdint.h>
#include <stddef.h>
#include <math.h>

#define ORACLE_BLOCK 64

/* ORACLE_MUTANT selects a deliberately wrong copy of one step, so that the pin
 * tests can show each such mistake is caught.  0 (the default) is the oracle. */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* IEEE 754 binary16 -> double, written out from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; exponent 0 is
 * subnormal (no implicit one, exponent -14), exponent 31 is inf/NaN. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);              /* frac * 2^-10 * 2^-14 */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25); /* (1 + frac/1024) * 2^(expo-15) */
    }
    return sign ? -v : v;
}

/* Section 4, step 1: per row, absmax -> scale -> int8 codes and per-64 row sums.
 * a_q: int8 [M][K]; s_a: fp32 [M]; rs: int32 [M][K/64]. */
void oracle_quant_pack(const float *x, long M, long K,
                       int8_t *a_q, float *s_a, int32_t *rs)
{
    long nb = K / ORACLE_BLOCK;
    for (long m = 0; m < M; ++m) {
        const float *row = x + m * K;
        float absmax = 0.0f;
        for (long k = 0; k < K; ++k) {
            float v = fabsf(row[k]);
            if (v > absmax) absmax = v;
        }
#if ORACLE_MUTANT == 6
        float scale = absmax / 128.0f;              /* mutant: wrong code range */
#else
        float scale = absmax / 127.0f;
#endif
        s_a[m] = scale;
        for (long k = 0; k < K; ++k) {
            int q = 0;
            /* A row whose scale is 0 -- absmax 0, or absmax / 127 below half the smallest
             * subnormal -- has no quotient to round; its codes are 0, as for a zero row. */
            if (scale > 0.0f) {
#if ORACLE_MUTANT == 5
                float r = rintf(row[k] / scale);    /* mutant: ties to even */
#else
                float r = roundf(row[k] / scale);
#endif
                if (r > 127.0f) r = 127.0f;
                if (r < -127.0f) r = -127.0f;
                q = (int)r;
            }
            a_q[m * K + k] = (int8_t)q;
        }
        for (long b = 0; b < nb; ++b) {
            int32_t sum = 0;
#if ORACLE_MUTANT == 4
            for (long i = 1; i < ORACLE_BLOCK; ++i) sum += a_q[m * K + b * ORACLE_BLOCK + i]; /* mutant */
#else
            for (long i = 0; i < ORACLE_BLOCK; ++i) sum += a_q[m * K + b * ORACLE_BLOCK + i];
#endif
            rs[m * nb + b] = sum;
        }
    }
}

/* Weight code q[n][k] from the packed byte stream. */
static int oracle_q(const uint8_t *wq, long K, long n, long k)
{
    uint8_t byte = wq[n * (K / 2) + k / 2];
#if ORACLE_MUTANT == 3
    return (k & 1) ? (byte & 0x0f) : (byte >> 4);   /* mutant: nibble order swapped */
#else
    return (k & 1) ? (byte >> 4) : (byte & 0x0f);
#endif
}

/* Per-block integer accumulators acc[m][n][b] = sum_{i in block b} a_q[m,i] q[n,i]
 * for the window rows m0..m0+mc-1, columns n0..n0+nc-1 (section 3, eq. (2), first sum). */
void oracle_block_acc(const int8_t *a_q, const uint8_t *wq, long M, long N, long K,
                      long m0, long mc, long n0, long nc, int32_t *acc)
{
    long nb = K / ORACLE_BLOCK;
    (void)M; (void)N;
    for (long mi = 0; mi < mc; ++mi)
        for (long ni = 0; ni < nc; ++ni)
            for (long b = 0; b < nb; ++b) {
                int32_t s = 0;
                for (long i = 0; i < ORACLE_BLOCK; ++i) {
                    long k = b * ORACLE_BLOCK + i;
                    s += (int32_t)a_q[(m0 + mi) * K + k] * oracle_q(wq, K, n0 + ni, k);
                }
                acc[(mi * nc + ni) * nb + b] = s;
            }
}

/* The same accumulators reached through section 3, eq. (3): the int8 activation is
 * split into a signed high nibble (arithmetic shift) and an unsigned low nibble,
 * and two 4-bit dot products are combined as 16 * hi_dot + lo_dot. */
void oracle_block_acc_nibble(const int8_t *a_q, const uint8_t *wq, long M, long N, long K,
                             long m0, long mc, long n0, long nc, int32_t *acc)
{
    long nb = K / ORACLE_BLOCK;
    (void)M; (void)N;
    for (long mi = 0; mi < mc; ++mi)
        for (long ni = 0; ni < nc; ++ni)
            for (long b = 0; b < nb; ++b) {
                int32_t hi_dot = 0, lo_dot = 0;
                for (long i = 0; i < ORACLE_BLOCK; ++i) {
                    long k = b * ORACLE_BLOCK + i;
                    int a = a_q[(m0 + mi) * K + k];
#if ORACLE_MUTANT == 8
                    int hi = (int)((unsigned)(a & 0xff) >> 4);   /* mutant: unsigned high nibble */
#else
                    int hi = a >> 4;          /* arithmetic shift: -8..7 */
#endif
                    int lo = a & 0x0f;        /* 0..15 */
                    int q = oracle_q(wq, K, n0 + ni, k);
                    hi_dot += hi * q;
                    lo_dot += lo * q;
                }
                acc[(mi * nc + ni) * nb + b] = 16 * hi_dot + lo_dot;
            }
}

/* Output for one row m (section 3, eq. (2), then section 4 step 3):
 *   y[m,n] = s_a[m] * sum_b s_w[n,b] * (acc[m,n,b] - z_w[n,b] * rs[m,b]) + bias[n]
 * in fp64.  bound[n] receives sum_b |s_a s_w (acc - z_w rs)|, the magnitude the
 * fp32 tolerance is stated against. */
static void oracle_linear_row(const int8_t *a_q, const float *s_a, const int32_t *rs,
                              const uint8_t *wq, const uint16_t *s_w, const uint16_t *z_w,
                              const float *bias, long N, long K, long m,
                              double *y_row, double *bound_row)
{
    long nb = K / ORACLE_BLOCK;
    for (long n = 0; n < N; ++n) {
        double total = 0.0, mag = 0.0;
        for (long b = 0; b < nb; ++b) {
            int64_t acc = 0;
            for (long i = 0; i < ORACLE_BLOCK; ++i) {
                long k = b * ORACLE_BLOCK + i;
                acc += (int64_t)a_q[m * K + k] * oracle_q(wq, K, n, k);
            }
#if ORACLE_MUTANT == 9
            double sw = oracle_half_to_double(z_w[n * nb + b]);   /* mutant: operands swapped */
            double zw = oracle_half_to_double(s_w[n * nb + b]);
#else
            double sw = oracle_half_to_double(s_w[n * nb + b]);
            double zw = oracle_half_to_double(z_w[n * nb + b]);
#endif
#if ORACLE_MUTANT == 1
            double term = sw * (double)acc;                        /* mutant: no zero point */
#elif ORACLE_MUTANT == 2
            double term = sw * ((double)acc + zw * (double)rs[m * nb + b]); /* mutant: sign */
#else
            double term = sw * ((double)acc - zw * (double)rs[m * nb + b]);
#endif
            total += term;
            mag += fabs((double)s_a[m] * term);
        }
#if ORACLE_MUTANT == 7
        y_row[n] = total + (bias ? (double)bias[n] : 0.0);          /* mutant: no s_a */
#elif ORACLE_MUTANT == 10
        y_row[n] = (double)s_a[m] * total;                          /* mutant: no bias */
#else
        y_row[n] = (double)s_a[m] * total + (bias ? (double)bias[n] : 0.0);
#endif
        if (bound_row) bound_row[n] = mag;
    }
}

/* y: fp64 [n_rows][N] for the listed rows (all rows when rows == NULL, n_rows == M).
 * bound: fp64 [n_rows][N] or NULL.  Rows run in parallel when built with OpenMP. */
void oracle_linear_rows(const int8_t *a_q, const float *s_a, const int32_t *rs,
                        const uint8_t *wq, const uint16_t *s_w, const uint16_t *z_w,
                        const float *bias, long M, long N, long K,
                        const long *rows, long n_rows, double *y, double *bound)
{
    (void)M;
#pragma omp parallel for schedule(dynamic, 1)
    for (long r = 0; r < n_rows; ++r) {
        long m = rows ? rows[r] : r;
        oracle_linear_row(a_q, s_a, rs, wq, s_w, z_w, bias, N, K, m,
                          y + r * N, bound ? bound + r * N : NULL);
    }
}

/* The whole prefill linear from fp32 activations, for the listed rows: section 4's
 * pre-pass (per row only, which is all the output needs) followed by the epilogue.
 * Scratch: a_q_row int8 [n_rows][K], rs_row int32 [n_rows][K/64], s_row fp32 [n_rows]
 * are caller-provided so this file allocates nothing. */
void oracle_prefill_linear_rows(const float *x, const uint8_t *wq, const uint16_t *s_w,
                                const uint16_t *z_w, const float *bias, long M, long N, long K,
                                const long *rows, long n_rows,
                                int8_t *a_q_rows, float *s_rows, int32_t *rs_rows,
                                double *y, double *bound)
{
    long nb = K / ORACLE_BLOCK;
    (void)M;
    for (long r = 0; r < n_rows; ++r) {
        long m = rows ? rows[r] : r;
        oracle_quant_pack(x + m * K, 1, K, a_q_rows + r * K, s_rows + r, rs_rows + r * nb);
    }
    oracle_linear_rows(a_q_rows, s_rows, rs_rows, wq, s_w, z_w, bias, n_rows, N, K,
                       NULL, n_rows, y, bound);
}

/* Number of OpenMP threads the parallel loops above use (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
