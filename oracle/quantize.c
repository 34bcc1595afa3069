/*
 * quantize.c — plain CPU reference for the FP8 and NVFP4 input encodings.
 *
 * TEST INFRASTRUCTURE ONLY (like oracle.c): loaded by the test suite, the
 * smoke check and the benchmark's CPU-baseline leg, never by the GPU library;
 * it shares no source with the CUDA path.
 *
 * What it computes (the formats of "ThunderKittens reaches 22.4 PFLOPS on
 * NVIDIA Rubin", NVFP4 and FP8 paragraphs: 8-bit floats with a per-tensor
 * scale; 4-bit floats with one 8-bit scale per 16 consecutive elements of a
 * row and one fp32 scale per tensor).  The pages give the formats, not the
 * recipe that picks the scales; the reading used throughout this project:
 *
 *   FP8 (e4m3):   amax = max |x| over the tensor
 *                 s    = 448 / amax                       (fp32 division)
 *                 q    = e4m3_rne_satfinite(x * s)        (fp32 product)
 *                 dequantisation scale = amax / 448       (what the GEMM takes)
 *                 amax = 0: s = 1, dequantisation scale 1.
 *   NVFP4:        g    = amax / (6 * 448)                 (fp32; 1 if amax = 0)
 *                 for each row and each block of 16 consecutive elements:
 *                   b    = max |x| over the block
 *                   sb   = e4m3_rne_satfinite(b / (6 * g))   (6*g rounded to fp32 first)
 *                   d    = dec(sb) * g                        (fp32 product)
 *                   q[i] = e2m1_rne_satfinite(x[i] / d), or 0 when d == 0
 *                 output: packed e2m1 (element 2j in the low nibble of byte
 *                 j), e4m3 block scales [rows][cols/16], g.
 *
 * Every decision that produces a code is taken in fp32 with a single IEEE
 * rounding per operation (multiply, divide), compiled with -ffp-contract=off.
 * Rounding to a format is round-to-nearest, ties to the even code, and values
 * beyond the largest finite magnitude saturate to it (448 for e4m3, 6 for
 * e2m1).  The sign of x is kept, also when the magnitude rounds to zero.
 * Inputs are finite (no NaN or infinity).
 */
#include <math.h>
#include <stdint.h>

/* e4m3 "fn": sign | exponent (4 bits, bias 7) | mantissa (3 bits).  Normal
 * values (1 + m/8) * 2^(e-7) for e = 1..15 except the NaN code e=15,m=7, so the
 * largest is 1.75 * 2^8 = 448; subnormals m/8 * 2^-6 = m * 2^-9.  Rounding is
 * done on the magnitude scaled to an integer number of units of the target
 * binade's spacing: nearbyint() under the default rounding mode rounds half to
 * even, and within one binade an even unit count is an even code. */
uint8_t oracle_e4m3_rne_sat(float x) {
    const uint8_t sign = signbit(x) ? 0x80u : 0x00u;
    double a = fabs((double)x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7Eu);
    if (a < ldexp(1.0, -6)) {                 /* subnormal range: spacing 2^-9 */
        const double m = nearbyint(a * 512.0); /* 0..8; 8 is the smallest normal */
        return (uint8_t)(sign | (uint8_t)m);   /* m = 8 -> exponent field 1, mantissa 0 */
    }
    int e2;
    (void)frexp(a, &e2);                      /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;                           /* a in [2^e, 2^(e+1)) */
    double units = nearbyint(ldexp(a, 3 - e)); /* in [8, 16]: spacing 2^(e-3) */
    if (units == 16.0) {
        units = 8.0;
        e += 1;
    }
    const int field = e + 7;                  /* 1..15 */
    const uint8_t code = (uint8_t)((field << 3) | ((int)units - 8));
    if ((code & 0x7Fu) > 0x7Eu) return (uint8_t)(sign | 0x7Eu); /* rounded past 448 */
    return (uint8_t)(sign | code);
}

/* e2m1: sign | exponent (2 bits, bias 1) | mantissa (1 bit): magnitudes
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6 for codes 0..7.  Same scheme: count units of the
 * binade's spacing (0.5 below 2, 1 in [2, 4), 2 in [4, 6]). */
uint8_t oracle_e2m1_rne_sat(float x) {
    const uint8_t sign = signbit(x) ? 0x8u : 0x0u;
    const double a = fabs((double)x);
    uint8_t code;
    if (a >= 6.0) {
        code = 7;
    } else if (a < 2.0) {
        code = (uint8_t)nearbyint(a * 2.0);       /* 0..4: 0, .5, 1, 1.5, 2 */
    } else if (a < 4.0) {
        code = (uint8_t)(nearbyint(a) + 2.0);     /* 4..6: 2, 3, 4 */
    } else {
        code = (uint8_t)(nearbyint(a * 0.5) + 4.0); /* 6..7: 4, 6 */
    }
    return (uint8_t)(sign | code);
}

static float dec_e4m3_value(uint8_t c) {
    const int e = (c >> 3) & 0xF, m = c & 7;
    const double v = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return (float)((c & 0x80) ? -v : v);
}

static float amax_of(const float* x, int64_t n) {
    float a = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        const float v = fabsf(x[i]);
        if (v > a) a = v;
    }
    return a;
}

/* x [rows][cols] fp32 row-major -> q [rows][cols] e4m3 codes; *dequant_scale. */
void oracle_quantize_fp8(int64_t rows, int64_t cols, const float* x, uint8_t* q, float* dequant_scale) {
    const int64_t n = rows * cols;
    const float amax = amax_of(x, n);
    const float s = amax > 0.0f ? 448.0f / amax : 1.0f;
    for (int64_t i = 0; i < n; ++i) {
        const float v = x[i] * s;
        q[i] = oracle_e4m3_rne_sat(v);
    }
    *dequant_scale = amax > 0.0f ? amax / 448.0f : 1.0f;
}

/* x [rows][cols] fp32 row-major, cols % 16 == 0 -> packed [rows][cols/2],
 * block scales sf [rows][cols/16] (e4m3), *g. */
void oracle_quantize_nvfp4(int64_t rows, int64_t cols, const float* x, uint8_t* packed, uint8_t* sf, float* g_out) {
    const float amax = amax_of(x, rows * cols);
    const float g = amax > 0.0f ? amax / 2688.0f : 1.0f;   /* 2688 = 6 * 448 */
    const float six_g = 6.0f * g;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < cols / 16; ++b) {
            const float* xb = x + r * cols + b * 16;
            const float bmax = amax_of(xb, 16);
            const float ratio = bmax / six_g;
            const uint8_t sb = oracle_e4m3_rne_sat(ratio);
            const float d = dec_e4m3_value(sb) * g;
            sf[r * (cols / 16) + b] = sb;
            uint8_t* out = packed + r * (cols / 2) + b * 8;
            for (int j = 0; j < 8; ++j) {
                uint8_t lo = 0, hi = 0;
                if (d != 0.0f) {
                    const float q0 = xb[2 * j] / d;
                    const float q1 = xb[2 * j + 1] / d;
                    lo = oracle_e2m1_rne_sat(q0);
                    hi = oracle_e2m1_rne_sat(q1);
                }
                out[j] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
    *g_out = g;
}
