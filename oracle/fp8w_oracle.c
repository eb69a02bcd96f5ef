/*
 * fp8w_oracle.c -- plain, slow CPU oracle for the FP8 weight-only linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library; it is written from the defining pages alone.
 *
 * What it computes (page "kadirnar/kernel-agent fp8-weights", section "The
 * contract"):
 *   scale[n] = amax_k |W[n,k]| / 448          (one fp32 IEEE division)
 *   q[n,k]   = e4m3( W[n,k] / scale[n] )      (round to nearest even, +-448)
 *   y[m,n]   = round_out( scale[n] * sum_k x[m,k] * e4m3val(q[n,k]) + bias[n] )
 *
 * Precision: the codes and scales are exact results (fp32 in, fp32/bytes
 * out); the linear layer is evaluated in fp64 with a sequential k-ascending
 * sum, then rounded once, directly from fp64, to bf16 or fp16.
 *
 * Build: plain C11, no fast-math, no FMA contraction (-ffp-contract=off), so
 * every float operation below is one IEEE operation on both x86-64 and Arm.
 *
 * Pins: every function here is checked by the test suite against values the
 * pages print, closed forms, exact rationals, invariants or brute force.
 * oracle_fp8_error's fields are named by the pages without definitions; its
 * readings are pinned by closed forms (crest of a one-spike row sqrt(k), of
 * a constant row 1; weights below half the smallest e4m3 step all
 * underflow; the error of a known tie) and invariances (power-of-two
 * rescaling, duplicated and permuted rows).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_ACT_BF16 1
#define ORACLE_ACT_F16 2

/* ------------------------------------------------------------------------ */
/* OCP E4M3 ("e4m3fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; no
 * infinities; only S.1111.111 is NaN, which leaves 1.75 * 2^8 = 448 as the
 * largest finite value.  Page "B04 Precision & Quantization", section 2,
 * "The numbers, derived rather than tabulated" (the E4M3 row and its
 * footnote on the NaN pattern).                                            */
/* ------------------------------------------------------------------------ */

double oracle_e4m3_decode(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 15;
    int m = b & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);            /* subnormal: m/8 * 2^(1-7) */
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Round-to-nearest-even into e4m3, saturating to +-448 ("satfinite").
 * Page "kadirnar/kernel-agent fp8-weights", "The contract" (round to nearest
 * even, clamped to +-448); page "tensormux Write an FP8 kernel", step 4 and
 * "Kernel design rules" (saturate rather than overflow).
 *
 * The rounding is done first on an unbounded e4m3 grid, then saturated.  On
 * that grid every value >= 448 rounds to 448 or above (the midpoint 464
 * between 448 and 480 ties to 448, whose mantissa is even), so after the
 * saturation every |v| >= 448 gives the code 0x7E.  The sign bit is kept for
 * zeros and for values that round to zero (IEEE sign rule).                */
uint8_t oracle_e4m3_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a;
    int ex, E;
    double r;
    if (isnan(v))
        return (uint8_t)(sign | 0x7F);
    a = fabs((double)v);                      /* exact */
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    if (a < 0.015625) {                       /* below 2^-6: step 2^-9 */
        r = nearbyint(ldexp(a, 9));           /* exact scaling, RNE, 0..8 */
        return (uint8_t)(sign | (uint8_t)r);  /* 8 -> 0x08, the min normal */
    }
    frexp(a, &ex);                            /* a = f * 2^ex, f in [0.5,1) */
    E = ex - 1;                               /* 2^E <= a < 2^(E+1), E in -6..8 */
    r = nearbyint(ldexp(a, 3 - E));           /* 8 .. 16, RNE */
    if (r == 16.0) {
        E += 1;
        r = 8.0;
    }
    return (uint8_t)(sign | (((E + 7) << 3) | ((int)r - 8)));
}

/* ------------------------------------------------------------------------ */
/* Per-output-channel scale and quantisation.                               */
/* ------------------------------------------------------------------------ */

/* scale = amax / 448 in fp32; an all-zero row (or an amax so small that the
 * quotient is 0) takes scale 1.0, so no division by zero can follow.  Page
 * "kadirnar/kernel-agent fp8-weights", "The contract"; the zero-row rule is
 * page "day98 quant_matmul.cu", quantizeSymmetric / quantizeColumns, and page
 * "tensormux Write an FP8 kernel", step 7 (handle scale = 0).               */
float oracle_row_scale(const float *row, int64_t k)
{
    float amax = 0.0f;
    float s;
    int64_t i;
    for (i = 0; i < k; ++i) {
        float a = fabsf(row[i]);
        if (a > amax)
            amax = a;
    }
    s = amax / 448.0f;
    if (s == 0.0f)
        s = 1.0f;
    return s;
}

/* W[n,k] row-major (nn.Linear [out, in]) -> codes[n,k], scales[n].
 * codes = e4m3(w / scale): an fp32 division, not a multiply by 1/scale.   */
void oracle_quantize(const float *w, int64_t n, int64_t k, uint8_t *codes,
                     float *scales)
{
    int64_t r, i;
    for (r = 0; r < n; ++r) {
        const float *row = w + r * k;
        float s = oracle_row_scale(row, k);
        scales[r] = s;
        for (i = 0; i < k; ++i) {
            float v = row[i] / s;
            codes[r * k + i] = oracle_e4m3_encode(v);
        }
    }
}

/* Per-group scales along K: one scale per run of g weights of a row (page
 * "B04 Precision & Quantization", section "Post-training quantization
 * versus quantization-aware training", the granularity table's per-group
 * row, g = 32/64/128).  Each group takes the per-channel rule on its own g
 * weights: scale = fp32(amax/448), 1.0 if that is 0, codes = e4m3 of the
 * fp32 quotient.  scales[n, k/g] row-major; k % g == 0.                   */
void oracle_quantize_grouped(const float *w, int64_t n, int64_t k, int64_t g,
                             uint8_t *codes, float *scales)
{
    int64_t r, j, i, ng = k / g;
    for (r = 0; r < n; ++r) {
        for (j = 0; j < ng; ++j) {
            const float *seg = w + r * k + j * g;
            float s = oracle_row_scale(seg, g);
            scales[r * ng + j] = s;
            for (i = 0; i < g; ++i)
                codes[r * k + j * g + i] = oracle_e4m3_encode(seg[i] / s);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* MX-style weight-only form: one E8M0 scale per 32 weights along K.  Page
 * "11. Inference with NVFP4/MXFP8", section "MXFP8-Style FP8": e4m3 codes
 * [N, K] and f8e8m0fnu scales [N, K/32], one scale per 32 values along K.
 * E8M0 ("e8m0fnu") is an unsigned biased exponent byte b, worth 2^(b-127);
 * 0xFF is NaN and there is no zero.
 *
 * The page fixes the storage, not how a block's scale is chosen.  Reading
 * taken: the per-channel rule limited to powers of two, i.e. the smallest
 * 2^e with 2^e >= amax/448, so that the block's largest weight maps to at
 * most 448 and is never clipped; amax 0 takes 2^0 (the per-channel rule's
 * 1.0); e is clamped to the format's [-127, 127]; an infinite amax has no
 * such power and takes the NaN scale, with every code of its block the
 * e4m3 NaN 0x7F.  Codes are e4m3(w / 2^e), one fp32 division as above.    */
/* ------------------------------------------------------------------------ */

#define ORACLE_MX_BLOCK 32

double oracle_e8m0_decode(uint8_t b)
{
    if (b == 0xFF)
        return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* The scale byte of a block of g weights: amax as in oracle_row_scale (NaN
 * weights do not count), then the exponent by exact comparisons in fp64
 * (448 * 2^e and amax are both exact there), from a first guess.          */
uint8_t oracle_mx_scale(const float *blk, int64_t g)
{
    float amax = 0.0f;
    int64_t i;
    int e;
    for (i = 0; i < g; ++i) {
        float a = fabsf(blk[i]);
        if (a > amax)
            amax = a;
    }
    if (isinf(amax))
        return 0xFF;
    if (amax == 0.0f)
        return 127;
    e = ilogb((double)amax) - 8;
    while (ldexp(448.0, e) < (double)amax)
        ++e;
    while (ldexp(448.0, e - 1) >= (double)amax)
        --e;
    if (e < -127)
        e = -127;
    if (e > 127)
        e = 127;
    return (uint8_t)(e + 127);
}

/* W[n,k] -> codes[n,k], scales[n, k/32] (E8M0 bytes); k % 32 == 0.        */
void oracle_quantize_mx(const float *w, int64_t n, int64_t k, uint8_t *codes,
                        uint8_t *scales)
{
    int64_t r, j, i, ng = k / ORACLE_MX_BLOCK;
    for (r = 0; r < n; ++r) {
        for (j = 0; j < ng; ++j) {
            const float *seg = w + r * k + j * ORACLE_MX_BLOCK;
            uint8_t *out = codes + r * k + j * ORACLE_MX_BLOCK;
            uint8_t b = oracle_mx_scale(seg, ORACLE_MX_BLOCK);
            scales[r * ng + j] = b;
            if (b == 0xFF) {
                memset(out, 0x7F, ORACLE_MX_BLOCK);
                continue;
            }
            {
                float s = (float)oracle_e8m0_decode(b);   /* exact, 2^-127 included */
                for (i = 0; i < ORACLE_MX_BLOCK; ++i)
                    out[i] = oracle_e4m3_encode(seg[i] / s);
            }
        }
    }
}

/* Dequantised weight in fp64: scale[n] * e4m3val(q[n,k]).  This is the
 * pages' fallback form q.float() * scale[:, None] ("The contract",
 * "Fallback").                                                              */
void oracle_dequantize(const uint8_t *codes, const float *scales, int64_t n,
                       int64_t k, double *wq)
{
    int64_t r, i;
    for (r = 0; r < n; ++r)
        for (i = 0; i < k; ++i)
            wq[r * k + i] = (double)scales[r] * oracle_e4m3_decode(codes[r * k + i]);
}

/* The same with per-group scales[n, k/g] (one per run of g codes of a row)
 * and with E8M0 scale bytes[n, k/32] (each worth 2^(b-127), 0xFF NaN):
 * scale times decoded code, exact in fp64.                                 */
void oracle_dequantize_grouped(const uint8_t *codes, const float *scales,
                               int64_t n, int64_t k, int64_t g, double *wq)
{
    int64_t r, i, ng = k / g;
    for (r = 0; r < n; ++r)
        for (i = 0; i < k; ++i)
            wq[r * k + i] = (double)scales[r * ng + i / g] * oracle_e4m3_decode(codes[r * k + i]);
}

void oracle_dequantize_mx(const uint8_t *codes, const uint8_t *scales, int64_t n,
                          int64_t k, double *wq)
{
    int64_t r, i, ng = k / ORACLE_MX_BLOCK;
    for (r = 0; r < n; ++r)
        for (i = 0; i < k; ++i)
            wq[r * k + i] = oracle_e8m0_decode(scales[r * ng + i / ORACLE_MX_BLOCK]) *
                            oracle_e4m3_decode(codes[r * k + i]);
}

/* ------------------------------------------------------------------------ */
/* Activation formats: bf16 (8 exponent, 7 mantissa bits, the top half of an
 * fp32) and fp16 (5 exponent bits, bias 15, 10 mantissa bits).  Page "B04",
 * section 2, the bf16 and fp16 rows.                                       */
/* ------------------------------------------------------------------------ */

double oracle_bf16_value(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oracle_f16_value(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double mag;
    if (e == 31)
        return m ? NAN : (sign ? -INFINITY : INFINITY);
    if (e == 0)
        mag = ldexp((double)m, -24);
    else
        mag = ldexp(1.0 + (double)m / 1024.0, e - 15);
    return sign ? -mag : mag;
}

/* Round an fp64 value to nearest-even on a binary grid with p significant
 * bits and smallest normal exponent emin (gradual underflow below it).
 * Returns the rounded magnitude as a double (exact), or +inf when the
 * rounded value exceeds maxfin.  Exact arithmetic: scaling by powers of two
 * and nearbyint() in the default round-to-nearest-even mode.              */
static double round_to_grid(double a, int p, int emin, double maxfin)
{
    int ex, e;
    double r, out;
    if (a == 0.0)
        return 0.0;
    frexp(a, &ex);
    e = ex - 1;                    /* 2^e <= a < 2^(e+1) */
    if (e < emin)
        e = emin;                  /* subnormal range: fixed quantum */
    r = nearbyint(ldexp(a, (p - 1) - e));
    out = ldexp(r, e - (p - 1));
    if (out > maxfin)
        return INFINITY;
    return out;
}

/* fp64 -> bf16 bits, one rounding straight from fp64 (no fp32 detour).  */
uint16_t oracle_round_bf16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a, r;
    float f;
    uint32_t u;
    if (isnan(v))
        return (uint16_t)(sign | 0x7FC0);
    a = fabs(v);
    r = round_to_grid(a, 8, -126, ldexp(255.0, 120)); /* max (2-2^-7)*2^127 */
    if (isinf(r))
        return (uint16_t)(sign | 0x7F80);
    f = (float)r;                  /* exact: r is a bf16 value */
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

/* fp64 -> fp16 bits, one rounding straight from fp64.                     */
uint16_t oracle_round_f16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a, r;
    int ex, e;
    if (isnan(v))
        return (uint16_t)(sign | 0x7E00);
    a = fabs(v);
    r = round_to_grid(a, 11, -14, 65504.0);
    if (isinf(r))
        return (uint16_t)(sign | 0x7C00);
    if (r == 0.0)
        return sign;
    if (r < ldexp(1.0, -14))       /* subnormal: r = t * 2^-24, t < 1024 */
        return (uint16_t)(sign | (uint16_t)ldexp(r, 24));
    frexp(r, &ex);
    e = ex - 1;
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) |
                      (uint16_t)(ldexp(r, 10 - e) - 1024.0));
}

static double act_value(const uint16_t *x, int act, int64_t idx)
{
    return act == ORACLE_ACT_F16 ? oracle_f16_value(x[idx]) : oracle_bf16_value(x[idx]);
}

/* ------------------------------------------------------------------------ */
/* The linear layer.  Page "kadirnar/kernel-agent fp8-weights", "The
 * contract": y[m,n] = scale[n] * sum_k x[m,k] q[n,k] + bias[n], scale and
 * bias applied once per output and one rounding to the activation dtype.
 * The reference pattern (fp64 plain loops, k ascending) is page "day98
 * quant_matmul.cu", matmulCpu.  bias may be NULL, meaning 0.              */
/* ------------------------------------------------------------------------ */

struct linear_job {
    const uint16_t *x;
    int act;
    int64_t m, k, n;
    const uint8_t *codes;
    const float *scales;
    const float *bias;
    uint16_t *y;
    double *yacc;
    int64_t n_begin, n_end;
    int64_t group;  /* 0: one scale per row; else scales[n, k/group] */
};

static void linear_range(const struct linear_job *j)
{
    int64_t mi, ni, ki;
    for (mi = 0; mi < j->m; ++mi) {
        for (ni = j->n_begin; ni < j->n_end; ++ni) {
            const uint8_t *q = j->codes + ni * j->k;
            double acc = 0.0, out;
            if (j->group == 0) {
                for (ki = 0; ki < j->k; ++ki)
                    acc += act_value(j->x, j->act, mi * j->k + ki) * oracle_e4m3_decode(q[ki]);
                out = (double)j->scales[ni] * acc;
            } else {
                /* each group's sum times its scale, groups in k order */
                int64_t gi, ng = j->k / j->group;
                out = 0.0;
                for (gi = 0; gi < ng; ++gi) {
                    acc = 0.0;
                    for (ki = gi * j->group; ki < (gi + 1) * j->group; ++ki)
                        acc += act_value(j->x, j->act, mi * j->k + ki) * oracle_e4m3_decode(q[ki]);
                    out += (double)j->scales[ni * ng + gi] * acc;
                }
            }
            out += j->bias ? (double)j->bias[ni] : 0.0;
            if (j->yacc)
                j->yacc[mi * j->n + ni] = out;
            if (j->y)
                j->y[mi * j->n + ni] = j->act == ORACLE_ACT_F16 ? oracle_round_f16(out)
                                                                : oracle_round_bf16(out);
        }
    }
}

static void *linear_thread(void *arg)
{
    linear_range((const struct linear_job *)arg);
    return NULL;
}

/* x[m,k] (bf16 or fp16 bits), codes[n,k], scales[n], bias[n] or NULL ->
 * y[m,n] (bits of the activation dtype) and, if yacc != NULL, the unrounded
 * fp64 value.  nthreads > 1 splits the output channels over POSIX threads;
 * each output is still one sequential sum, so the result does not depend
 * on the thread count.  Returns 0, or -1 if a thread could not start.     */
static int linear_run(const uint16_t *x, int act, int64_t m, int64_t k,
                      const uint8_t *codes, const float *scales, int64_t group,
                      const float *bias, int64_t n, uint16_t *y, double *yacc,
                      int nthreads)
{
    struct linear_job *jobs;
    pthread_t *tids;
    int t, started = 0, rc = 0;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > n)
        nthreads = (int)(n > 0 ? n : 1);
    jobs = (struct linear_job *)calloc((size_t)nthreads, sizeof *jobs);
    tids = (pthread_t *)calloc((size_t)nthreads, sizeof *tids);
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return -1;
    }
    for (t = 0; t < nthreads; ++t) {
        struct linear_job *j = &jobs[t];
        j->x = x; j->act = act; j->m = m; j->k = k; j->n = n;
        j->codes = codes; j->scales = scales; j->bias = bias;
        j->y = y; j->yacc = yacc; j->group = group;
        j->n_begin = n * t / nthreads;
        j->n_end = n * (t + 1) / nthreads;
    }
    if (nthreads == 1) {
        linear_range(&jobs[0]);
    } else {
        for (t = 0; t < nthreads; ++t) {
            if (pthread_create(&tids[t], NULL, linear_thread, &jobs[t]) != 0) {
                rc = -1;
                break;
            }
            ++started;
        }
        for (t = 0; t < started; ++t)
            pthread_join(tids[t], NULL);
        /* a thread that failed to start leaves its range to this thread */
        for (t = started; t < nthreads; ++t)
            linear_range(&jobs[t]);
        rc = 0;
    }
    free(jobs);
    free(tids);
    return rc;
}

int oracle_linear(const uint16_t *x, int act, int64_t m, int64_t k,
                  const uint8_t *codes, const float *scales, const float *bias,
                  int64_t n, uint16_t *y, double *yacc, int nthreads)
{
    return linear_run(x, act, m, k, codes, scales, 0, bias, n, y, yacc, nthreads);
}

/* The same with per-group scales[n, k/g]:
 * y[m,n] = RN_act( sum_j scale[n,j] * sum_{k in group j} x[m,k] q[n,k] + bias[n] ),
 * fp64 throughout, one rounding.                                           */
int oracle_linear_grouped(const uint16_t *x, int act, int64_t m, int64_t k,
                          const uint8_t *codes, const float *scales, int64_t g,
                          const float *bias, int64_t n, uint16_t *y, double *yacc,
                          int nthreads)
{
    return linear_run(x, act, m, k, codes, scales, g, bias, n, y, yacc, nthreads);
}

/* The MX-style form: the per-group linear layer with g = 32 and each scale
 * the value of its E8M0 byte (exact in fp32, 2^-127 included; 0xFF is NaN).
 * Returns 0, or -1 if memory or a thread could not be had.               */
int oracle_linear_mx(const uint16_t *x, int act, int64_t m, int64_t k,
                     const uint8_t *codes, const uint8_t *scales,
                     const float *bias, int64_t n, uint16_t *y, double *yacc,
                     int nthreads)
{
    int64_t i, ns = n * (k / ORACLE_MX_BLOCK);
    int rc;
    float *sf = (float *)malloc((size_t)(ns > 0 ? ns : 1) * sizeof *sf);
    if (!sf)
        return -1;
    for (i = 0; i < ns; ++i)
        sf[i] = (float)oracle_e8m0_decode(scales[i]);
    rc = linear_run(x, act, m, k, codes, sf, ORACLE_MX_BLOCK, bias, n, y, yacc, nthreads);
    free(sf);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* W8A8: activations quantised too (page "tensormux Write an FP8 kernel",
 * steps 2-4 and its epilogue: per-token activation scales, per-channel
 * weight scales, both amax / 448, and the accumulator multiplied by both;
 * page "kadirnar/kernel-agent fp8-weights" calls this a different target
 * from weight-only).  Activation codes qx[m, k] and scales sx[m] come from
 * the per-row rule above applied to the activations widened to fp32.
 *   y[m,n] = RN_out( sx[m] * sw[n] * sum_k e4m3(qx[m,k]) e4m3(qw[n,k]) + bias[n] )
 * in fp64 (every product and the k-ascending sum exact to fp64 rounding),
 * one rounding to the output type (bf16 or fp16).                         */
/* ------------------------------------------------------------------------ */
int oracle_linear_w8a8(const uint8_t *qx, const float *sx, int act, int64_t m,
                       int64_t k, const uint8_t *qw, const float *sw,
                       const float *bias, int64_t n, uint16_t *y, double *yacc)
{
    int64_t mi, ni, ki;
    for (mi = 0; mi < m; ++mi) {
        for (ni = 0; ni < n; ++ni) {
            double acc = 0.0, out;
            for (ki = 0; ki < k; ++ki)
                acc += oracle_e4m3_decode(qx[mi * k + ki]) * oracle_e4m3_decode(qw[ni * k + ki]);
            out = (double)sx[mi] * (double)sw[ni] * acc + (bias ? (double)bias[ni] : 0.0);
            if (yacc)
                yacc[mi * n + ni] = out;
            if (y)
                y[mi * n + ni] = act == ORACLE_ACT_F16 ? oracle_round_f16(out) : oracle_round_bf16(out);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Weight error report, the fields of fp8_error(weight, q, scale) named on
 * page "kadirnar/kernel-agent fp8-weights", "The contract".  The page names
 * the fields but prints no definitions; the readings used here:
 *   out[0] rel_l2               ||W - Wq||_F / ||W||_F
 *   out[1] worst_channel_rel_l2 max over rows with ||W_n|| > 0 of ||W_n - Wq_n|| / ||W_n||
 *   out[2] underflow            share of nonzero w whose code decodes to 0
 *   out[3] crest                max over nonzero rows of amax_n / rms_n
 * with Wq = scale[n] * e4m3val(q).  Sums in fp64.                          */
/* ------------------------------------------------------------------------ */
void oracle_fp8_error(const float *w, int64_t n, int64_t k, const uint8_t *codes,
                      const float *scales, double *out)
{
    double num = 0.0, den = 0.0, worst = 0.0, crest = 0.0;
    int64_t nonzero = 0, under = 0, r, i;
    for (r = 0; r < n; ++r) {
        double rn = 0.0, rd = 0.0, amax = 0.0;
        for (i = 0; i < k; ++i) {
            double wv = (double)w[r * k + i];
            double qv = oracle_e4m3_decode(codes[r * k + i]);
            double d = wv - (double)scales[r] * qv;
            rn += d * d;
            rd += wv * wv;
            if (fabs(wv) > amax)
                amax = fabs(wv);
            if (wv != 0.0) {
                ++nonzero;
                if (qv == 0.0)
                    ++under;
            }
        }
        num += rn;
        den += rd;
        if (rd > 0.0) {
            double rel = sqrt(rn / rd);
            double c = amax / sqrt(rd / (double)k);
            if (rel > worst)
                worst = rel;
            if (c > crest)
                crest = c;
        }
    }
    out[0] = den > 0.0 ? sqrt(num / den) : 0.0;
    out[1] = worst;
    out[2] = nonzero ? (double)under / (double)nonzero : 0.0;
    out[3] = crest;
}

/* Bulk helpers so that tests can sweep many values in one call. */
void oracle_e4m3_encode_many(const float *v, int64_t count, uint8_t *out)
{
    int64_t i;
    for (i = 0; i < count; ++i)
        out[i] = oracle_e4m3_encode(v[i]);
}

void oracle_round_bf16_many(const double *v, int64_t count, uint16_t *out)
{
    int64_t i;
    for (i = 0; i < count; ++i)
        out[i] = oracle_round_bf16(v[i]);
}

void oracle_round_f16_many(const double *v, int64_t count, uint16_t *out)
{
    int64_t i;
    for (i = 0; i < count; ++i)
        out[i] = oracle_round_f16(v[i]);
}
