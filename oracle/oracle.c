/*
 * oracle.c -- plain, slow CPU reference for the fused
 * "reduce R partials + residual add + RMSNorm (+ per-group FP8 quant)" epilogue.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library; the two meet only in the seeded input arrays.
 *
 * What it computes, per token row t (all names follow the pages):
 *
 *   x_hat[h]        = (((f32(P0[t,h]) + f32(P1[t,h])) + ...) + f32(P[R-1][t,h]))
 *                     + f32(residual[t,h])            fp32 adds, rank order, residual last
 *   residual_out[h] = bf16_rn(x_hat[h])
 *   x[h]            = residual_out[h]                 (exactly representable in fp64)
 *   rstd            = 1 / sqrt( (sum_h x[h]^2) / H + eps )      in fp64
 *   y[h]            = bf16_rn( x[h] * rstd * gamma[h] )         in fp64, one rounding
 *
 * Sources:
 *  - "ROCm AITER fused all-reduce + RMSNorm" (vLLM PR 37646 summary), section
 *    "key source snippets", allreduce_rms_fusion.py: the replaced subgraph is
 *    allreduce_output = all_reduce(input); rms = rms_norm(allreduce_output, weight, eps);
 *    and the pattern returns (rms, allreduce_output).  The fused-add variant
 *    (fused_add_rms_norm) adds the residual before the norm (implementation
 *    breakdown, item 2).
 *  - "AMD fused AllReduce-RMSNorm quant kernel" (SGLang PR 24651 summary),
 *    section "key source snippets", layernorm.py: the two-kernel tier quantises
 *    fused_out[0] -- the normalised bf16 activation -- per 1x128 group; the
 *    single-kernel tier returns ((fp8, scale), residual) or
 *    ((bf16, fp8, scale), residual) when keep_bf16 is set.
 *
 * Readings where the pages are silent (each one is listed with its reason in
 * the design notes):
 *  - the sum is fp32 in rank order 0..R-1, the residual added last, one RNE to
 *    bf16; the norm reads the bf16-rounded residual_out;
 *  - RMSNorm is x * rsqrt(mean(x^2) + eps) * gamma, eps inside the root
 *    ("variance_epsilon"), no (1 + gamma) offset, gamma bf16 [H];
 *  - a NULL residual is a row of +0.0;
 *  - per-group quant: a = max |y| over the group, s = fp32(a / 448),
 *    q = e4m3fn_rn_satfinite(fp32(y / s)), both divisions IEEE fp32 (the
 *    precision the kernel decides the code in); s == 0 gives q = 0;
 *  - scales are [T, H/group] row-major fp32; e4m3 is the OCP "fn" format
 *    (bias 7, max 448, no infinities, NaN = S.1111.111);
 *  - the MXFP4 output (a third fused variant the AITER fix names without a
 *    format) follows the OCP Microscaling Formats v1.0 conversion: blocks of
 *    32, shared E8M0 exponent floor(log2(absmax)) - 2, E2M1 elements rounded
 *    to nearest even and saturated; element 2i in the low nibble of a byte.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -fopenmp -shared -fPIC.
 * ffp-contract=off keeps every fp32 add a separately rounded IEEE add.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <fenv.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Number formats, written from their bit-level definitions.                */
/* ------------------------------------------------------------------------ */

/* Round a non-negative finite value to a binary floating-point grid with
 * p significand bits (implicit bit included) and minimum normal exponent emin,
 * round-to-nearest, ties to even.  Below 2^emin the grid spacing stays at
 * 2^(emin - p + 1) (gradual underflow).  No upper clamp here. */
static double round_to_grid(double a, int p, int emin)
{
    if (a == 0.0) return 0.0;
    int ex;
    (void)frexp(a, &ex);              /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;                   /* exponent of the leading bit */
    if (e < emin) e = emin;
    double ulp = ldexp(1.0, e - (p - 1));
    double n = nearbyint(a / ulp);    /* exact scaling; FE_TONEAREST = ties to even */
    return n * ulp;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_double(uint16_t b)
{
    int s = (b >> 15) & 1;
    int e = (b >> 7) & 0xFF;
    int m = b & 0x7F;
    double v;
    if (e == 0xFF) v = (m == 0) ? INFINITY : NAN;
    else if (e == 0) v = ldexp((double)m, -126 - 7);
    else v = ldexp(128.0 + (double)m, e - 127 - 7);
    return s ? -v : v;
}

uint16_t oracle_bf16_from_double(double v)
{
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    const double max_finite = ldexp(255.0, 127 - 7);  /* (2 - 2^-7) * 2^127 */
    if (isinf(a)) return sign | 0x7F80;
    double r = round_to_grid(a, 8, -126);
    if (r > max_finite) return sign | 0x7F80;         /* RNE overflow -> inf */
    if (r == 0.0) return sign;
    int ex;
    (void)frexp(r, &ex);
    int e = ex - 1;
    if (e < -126) {                                    /* subnormal: r = m * 2^-133 */
        return sign | (uint16_t)(int)ldexp(r, 133);
    }
    int m = (int)ldexp(r, 7 - e) - 128;               /* r = (128 + m) * 2^(e-7) */
    if (m == 128) { m = 0; e += 1; }
    return sign | (uint16_t)((e + 127) << 7) | (uint16_t)m;
}

/* OCP 8-bit floating point, E4M3 ("fn"): bias 7, exponent field 1..15 normal,
 * S.1111.111 is NaN, no infinities, max finite S.1111.110 = 448, min normal
 * 2^-6, subnormals m/8 * 2^-6. */
double oracle_e4m3_to_double(uint8_t c)
{
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7) v = NAN;
    else if (e == 0) v = ldexp((double)m, -6 - 3);
    else v = ldexp(8.0 + (double)m, e - 7 - 3);
    return s ? -v : v;
}

/* Round to nearest even, saturate to +-448 (satfinite: overflow and +-inf
 * clamp to the largest finite value; NaN maps to the NaN code). */
uint8_t oracle_e4m3_from_double(double v)
{
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0;
    double a = fabs(v);
    double r = isinf(a) ? 448.0 : round_to_grid(a, 4, -6);
    if (r > 448.0) r = 448.0;
    if (r == 0.0) return sign;
    if (r < ldexp(1.0, -6)) {                          /* subnormal: r = m * 2^-9 */
        return sign | (uint8_t)(int)ldexp(r, 9);
    }
    int ex;
    (void)frexp(r, &ex);
    int e = ex - 1;                                    /* -6 .. 8 */
    int m = (int)ldexp(r, 3 - e) - 8;                  /* r = (8 + m) * 2^(e-3) */
    return sign | (uint8_t)((e + 7) << 3) | (uint8_t)m;
}

/* OCP Microscaling (MX) v1.0 FP4 element type E2M1: 1 sign bit, 2 exponent
 * bits (bias 1), 1 mantissa bit; exponent field 0 holds zero and the subnormal
 * 0.5; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; no infinities, no NaN. */
double oracle_e2m1_to_double(uint8_t c)
{
    int s = (c >> 3) & 1;
    int e = (c >> 1) & 0x3;
    int m = c & 0x1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* Round to nearest even on the E2M1 grid, saturating to +-6. */
uint8_t oracle_e2m1_from_double(double v)
{
    uint8_t sign = signbit(v) ? 0x8 : 0;
    double a = fabs(v);
    double r = (isnan(v) || isinf(a)) ? 6.0 : round_to_grid(a, 2, 0);
    if (r > 6.0) r = 6.0;
    if (r == 0.0) return sign;
    if (r < 1.0) return sign | 0x1;                    /* 0.5: subnormal */
    int ex;
    (void)frexp(r, &ex);
    int e = ex - 1;                                    /* 0 .. 2 */
    int m = (int)ldexp(r, 1 - e) - 2;                  /* r = (2 + m) * 2^(e-1) */
    return sign | (uint8_t)((e + 1) << 1) | (uint8_t)m;
}

/* MX scale type E8M0: 2^(code - 127); code 0xFF is NaN. */
double oracle_e8m0_to_double(uint8_t c)
{
    return c == 0xFF ? NAN : ldexp(1.0, (int)c - 127);
}

static inline float bf16_to_f32(uint16_t b) { return (float)oracle_bf16_to_double(b); }

/* ------------------------------------------------------------------------ */
/* The epilogue.                                                             */
/* ------------------------------------------------------------------------ */

/* One token row.  partials: [R][T][H] contiguous, row t of partial r at
 * partials + (r*T + t)*H. */
static void reduce_rmsnorm_row(const uint16_t* partials, int R, int64_t T,
                               const uint16_t* residual, const uint16_t* gamma,
                               int H, float eps, int64_t t,
                               uint16_t* residual_out, uint16_t* y)
{
    uint16_t* ro = residual_out + t * (int64_t)H;
    /* Reduce: fp32, rank order, residual last. */
    for (int h = 0; h < H; ++h) {
        float acc = bf16_to_f32(partials[((int64_t)0 * T + t) * H + h]);
        for (int r = 1; r < R; ++r) {
            float p = bf16_to_f32(partials[((int64_t)r * T + t) * H + h]);
            acc = acc + p;
        }
        float res = residual ? bf16_to_f32(residual[t * (int64_t)H + h]) : 0.0f;
        acc = acc + res;
        ro[h] = oracle_bf16_from_double((double)acc);
    }
    if (!y) return;
    /* RMSNorm of the bf16 residual_out, in fp64. */
    double ss = 0.0;
    for (int h = 0; h < H; ++h) {
        double x = oracle_bf16_to_double(ro[h]);
        ss += x * x;
    }
    double rstd = 1.0 / sqrt(ss / (double)H + (double)eps);
    uint16_t* yo = y + t * (int64_t)H;
    for (int h = 0; h < H; ++h) {
        double x = oracle_bf16_to_double(ro[h]);
        double g = oracle_bf16_to_double(gamma[h]);
        yo[h] = oracle_bf16_from_double(x * rstd * g);
    }
}

/* Returns 0 on success, -1 on a bad argument.  y may be NULL (residual_out
 * only).  threads <= 1 runs serially; threads > 1 splits rows over OpenMP
 * threads (each row is computed exactly as in the serial loop). */
int oracle_reduce_rmsnorm(const uint16_t* partials, int R, const uint16_t* residual,
                          const uint16_t* gamma, int64_t T, int H, float eps,
                          uint16_t* residual_out, uint16_t* y, int threads)
{
    if (R < 1 || T < 0 || H < 1 || !partials || !residual_out) return -1;
    if (y && !gamma) return -1;
    if (fegetround() != FE_TONEAREST) return -1;
#ifdef _OPENMP
    if (threads > 1) {
        #pragma omp parallel for num_threads(threads) schedule(static)
        for (int64_t t = 0; t < T; ++t)
            reduce_rmsnorm_row(partials, R, T, residual, gamma, H, eps, t, residual_out, y);
        return 0;
    }
#else
    (void)threads;
#endif
    for (int64_t t = 0; t < T; ++t)
        reduce_rmsnorm_row(partials, R, T, residual, gamma, H, eps, t, residual_out, y);
    return 0;
}

/* Per-group dynamic FP8 quant of a bf16 [T][H] activation.
 * q: [T][H] e4m3fn codes; scales: [T][H/group] fp32, row-major. */
static void quant_row(const uint16_t* y, int H, int group, int64_t t,
                      uint8_t* q, float* scales)
{
    int ngroups = H / group;
    for (int g = 0; g < ngroups; ++g) {
        const uint16_t* yg = y + t * (int64_t)H + (int64_t)g * group;
        uint8_t* qg = q + t * (int64_t)H + (int64_t)g * group;
        float a = 0.0f;
        for (int i = 0; i < group; ++i) {
            float v = fabsf(bf16_to_f32(yg[i]));
            if (v > a) a = v;
        }
        float s = a / 448.0f;                          /* IEEE fp32 divide */
        scales[t * (int64_t)ngroups + g] = s;
        for (int i = 0; i < group; ++i) {
            if (s == 0.0f) { qg[i] = 0; continue; }
            float v = bf16_to_f32(yg[i]) / s;          /* IEEE fp32 divide */
            qg[i] = oracle_e4m3_from_double((double)v);
        }
    }
}

int oracle_quant_per_group(const uint16_t* y, int64_t T, int H, int group,
                           uint8_t* q, float* scales, int threads)
{
    if (!y || !q || !scales || T < 0 || group < 1 || H < group || H % group) return -1;
    if (fegetround() != FE_TONEAREST) return -1;
#ifdef _OPENMP
    if (threads > 1) {
        #pragma omp parallel for num_threads(threads) schedule(static)
        for (int64_t t = 0; t < T; ++t) quant_row(y, H, group, t, q, scales);
        return 0;
    }
#else
    (void)threads;
#endif
    for (int64_t t = 0; t < T; ++t) quant_row(y, H, group, t, q, scales);
    return 0;
}

/* MXFP4 (OCP MX v1.0: block size 32, E8M0 scale, E2M1 elements) of a bf16
 * [T][H] activation, blocks of 32 consecutive elements along H:
 *   shared_exp = floor(log2(max |y| over the block)) - 2   (2 = emax of E2M1),
 *                clamped to the E8M0 range [-127, 127];
 *   X = 2^shared_exp;  P_i = e2m1_rn_satfinite(y_i / X).
 * An all-zero block gets scale code 0 (2^-127) and zero elements.
 * q: [T][H/2] bytes, element 2i in the low nibble; scales: [T][H/32] E8M0. */
static void mxfp4_row(const uint16_t* y, int H, int64_t t, uint8_t* q, uint8_t* scales)
{
    int nb = H / 32;
    for (int b = 0; b < nb; ++b) {
        const uint16_t* yb = y + t * (int64_t)H + (int64_t)b * 32;
        double amax = 0.0;
        for (int i = 0; i < 32; ++i) {
            double v = fabs(oracle_bf16_to_double(yb[i]));
            if (v > amax) amax = v;
        }
        int shared_exp = -127;
        if (amax > 0.0) {
            int ex;
            (void)frexp(amax, &ex);                    /* amax = f * 2^ex, f in [0.5, 1) */
            shared_exp = (ex - 1) - 2;
            if (shared_exp < -127) shared_exp = -127;
            if (shared_exp > 127) shared_exp = 127;
        }
        scales[t * (int64_t)nb + b] = (uint8_t)(shared_exp + 127);
        uint8_t* qb = q + t * (int64_t)(H / 2) + (int64_t)b * 16;
        for (int i = 0; i < 16; ++i) {
            uint8_t lo = 0, hi = 0;
            if (amax > 0.0) {
                lo = oracle_e2m1_from_double(ldexp(oracle_bf16_to_double(yb[2 * i]), -shared_exp));
                hi = oracle_e2m1_from_double(ldexp(oracle_bf16_to_double(yb[2 * i + 1]), -shared_exp));
            }
            qb[i] = (uint8_t)(lo | (hi << 4));
        }
    }
}

int oracle_mxfp4(const uint16_t* y, int64_t T, int H, uint8_t* q, uint8_t* scales, int threads)
{
    if (!y || !q || !scales || T < 0 || H < 32 || H % 32) return -1;
    if (fegetround() != FE_TONEAREST) return -1;
#ifdef _OPENMP
    if (threads > 1) {
        #pragma omp parallel for num_threads(threads) schedule(static)
        for (int64_t t = 0; t < T; ++t) mxfp4_row(y, H, t, q, scales);
        return 0;
    }
#else
    (void)threads;
#endif
    for (int64_t t = 0; t < T; ++t) mxfp4_row(y, H, t, q, scales);
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
