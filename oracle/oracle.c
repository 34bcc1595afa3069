/*
 * oracle.c — plain, slow CPU reference for the dense tiled GEMM C = A·Bᵀ.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code; the GPU library never does.
 * It shares no source with the CUDA path.
 *
 * What it computes (the plain definition the tiled kernels reach faster):
 *
 *   acc[m][n] = sum_{k=0}^{K-1} dec(A[m][k]) * dec(B[n][k])
 *
 * accumulated in fp32, in increasing k, each product rounded to fp32 and then
 * added (no fused multiply-add; build with -ffp-contract=off, never
 * -ffast-math).  This is the operation the ThunderKittens pages call mma_ABt
 * ("att += Q @ K^T", paper summary, "PyTorch-Like Operations on Tiles") with
 * bf16 inputs and an fp32 accumulator ("Warp-Level: Tile Operations", App. B.1
 * GEMM walk-through).  Output formats:
 *
 *   bf16 :  C = bf16_rne(acc)
 *   fp8  :  C = bf16_rne((acc * scale_a) * scale_b)          (e4m3 operands)
 *   nvfp4:  C = bf16_rne((acc * g_a) * g_b), with dec(A[m][k]) =
 *           e2m1(A[m][k]) * e4m3(SFA[m][k/16]) formed in fp32 (exact), same
 *           for B (block-scaled 4-bit, Rubin article, NVFP4 paragraph).
 *
 * Decoding is by table, built here from the format bit-field definitions:
 *   bf16 : fp32 bits = h << 16
 *   e4m3 : sign | 4-bit exponent (bias 7) | 3-bit mantissa; exponent 0 is
 *          subnormal (m/8 * 2^-6); 0x7F / 0xFF are NaN; no infinities.
 *   e2m1 : sign | 2-bit exponent (bias 1) | 1-bit mantissa; exponent 0 is
 *          subnormal (m * 0.5).
 * FP4 packing: element 2j in the low nibble of byte j, 2j+1 in the high nibble.
 *
 * Rows of the output are independent; OpenMP splits them across host cores.
 * That changes nothing in the arithmetic of any single output element.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static float g_e4m3[256];
static float g_e2m1[16];
static int g_ready = 0;

static void build_tables(void) {
    for (int code = 0; code < 256; ++code) {
        int s = (code >> 7) & 1, e = (code >> 3) & 0xF, m = code & 7;
        float v;
        if (e == 0xF && m == 7) {
            v = NAN;
        } else if (e == 0) {
            v = ldexpf((float)m / 8.0f, 1 - 7);
        } else {
            v = ldexpf(1.0f + (float)m / 8.0f, e - 7);
        }
        g_e4m3[code] = s ? -v : v;
    }
    for (int code = 0; code < 16; ++code) {
        int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
        float v = (e == 0) ? 0.5f * (float)m : ldexpf(1.0f + 0.5f * (float)m, e - 1);
        g_e2m1[code] = s ? -v : v;
    }
    g_ready = 1;
}

void oracle_init(void) {
    if (!g_ready) build_tables();
}

float oracle_dec_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

float oracle_dec_e4m3(uint8_t c) {
    oracle_init();
    return g_e4m3[c];
}

float oracle_dec_e2m1(uint8_t c) {
    oracle_init();
    return g_e2m1[c & 0xF];
}

/* Round an fp32 to the nearest bf16, ties to even.  Of the two bf16 values
 * that bracket f (its upper 16 bits, and that plus one ulp) pick the nearer;
 * on an exact tie pick the one whose last bit is 0.  NaN stays NaN (quiet). */
uint16_t oracle_rne_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lower = u >> 16;          /* truncated candidate        */
    uint32_t rest = u & 0xFFFFu;       /* discarded low half          */
    if (rest > 0x8000u || (rest == 0x8000u && (lower & 1u))) lower += 1u;
    return (uint16_t)lower;
}

/* ---- decoders (whole arrays) ------------------------------------------ */

void oracle_decode_bf16(const uint16_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_dec_bf16(in[i]);
}

void oracle_decode_e4m3(const uint8_t* in, float* out, int64_t n) {
    oracle_init();
    for (int64_t i = 0; i < n; ++i) out[i] = g_e4m3[in[i]];
}

/* packed [rows][K/2] e2m1 with e4m3 block scales [rows][K/16] -> fp32 [rows][K] */
void oracle_decode_nvfp4(const uint8_t* packed, const uint8_t* sf, float* out, int64_t rows, int64_t K) {
    oracle_init();
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t k = 0; k < K; ++k) {
            uint8_t byte = packed[r * (K / 2) + k / 2];
            uint8_t nib = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            float scale = g_e4m3[sf[r * (K / 16) + k / 16]];
            out[r * K + k] = g_e2m1[nib] * scale;
        }
    }
}

/* ---- the reference contraction ----------------------------------------- */

/* acc[i][n] = sum_k Ad[i][k] * Bd[n][k] in fp32, k ascending, for the nrows
 * decoded rows of A given in Ad ([nrows][K]) against all N rows of Bd. */
static void contract_f32(const float* Ad, const float* Bd, int64_t nrows, int64_t N, int64_t K, float* acc) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        const float* a = Ad + i * K;
        for (int64_t n = 0; n < N; ++n) {
            const float* b = Bd + n * K;
            float s = 0.0f;
            for (int64_t k = 0; k < K; ++k) {
                float p = a[k] * b[k];
                s = s + p;
            }
            acc[i * N + n] = s;
        }
    }
}

static void finish_bf16(const float* acc, int64_t count, float sa, float sb, int scaled, uint16_t* C) {
    for (int64_t i = 0; i < count; ++i) {
        float v = acc[i];
        if (scaled) {
            v = v * sa;
            v = v * sb;
        }
        C[i] = oracle_rne_bf16(v);
    }
}

/* Row-subset forms: rows == NULL means all M rows (nrows must equal M then).
 * acc and C are [nrows][N]; either may be NULL.  Return 0 on success. */

int oracle_gemm_bf16_rows(int64_t M, int64_t N, int64_t K, const uint16_t* A, const uint16_t* B,
                          const int64_t* rows, int64_t nrows, float* acc, uint16_t* C) {
    (void)M;
    float* Ad = (float*)malloc(sizeof(float) * (size_t)(nrows * K));
    float* Bd = (float*)malloc(sizeof(float) * (size_t)(N * K));
    float* tmp = acc ? acc : (float*)malloc(sizeof(float) * (size_t)(nrows * N));
    if (!Ad || !Bd || !tmp) return 1;
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        oracle_decode_bf16(A + r * K, Ad + i * K, K);
    }
    oracle_decode_bf16(B, Bd, N * K);
    contract_f32(Ad, Bd, nrows, N, K, tmp);
    if (C) finish_bf16(tmp, nrows * N, 1.0f, 1.0f, 0, C);
    free(Ad);
    free(Bd);
    if (!acc) free(tmp);
    return 0;
}

int oracle_gemm_fp8_rows(int64_t M, int64_t N, int64_t K, const uint8_t* A, const uint8_t* B, float scale_a,
                         float scale_b, const int64_t* rows, int64_t nrows, float* acc, uint16_t* C) {
    (void)M;
    float* Ad = (float*)malloc(sizeof(float) * (size_t)(nrows * K));
    float* Bd = (float*)malloc(sizeof(float) * (size_t)(N * K));
    float* tmp = acc ? acc : (float*)malloc(sizeof(float) * (size_t)(nrows * N));
    if (!Ad || !Bd || !tmp) return 1;
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        oracle_decode_e4m3(A + r * K, Ad + i * K, K);
    }
    oracle_decode_e4m3(B, Bd, N * K);
    contract_f32(Ad, Bd, nrows, N, K, tmp);
    if (C) finish_bf16(tmp, nrows * N, scale_a, scale_b, 1, C);
    free(Ad);
    free(Bd);
    if (!acc) free(tmp);
    return 0;
}

int oracle_gemm_nvfp4_rows(int64_t M, int64_t N, int64_t K, const uint8_t* A, const uint8_t* B, const uint8_t* SFA,
                           const uint8_t* SFB, float g_a, float g_b, const int64_t* rows, int64_t nrows, float* acc,
                           uint16_t* C) {
    (void)M;
    float* Ad = (float*)malloc(sizeof(float) * (size_t)(nrows * K));
    float* Bd = (float*)malloc(sizeof(float) * (size_t)(N * K));
    float* tmp = acc ? acc : (float*)malloc(sizeof(float) * (size_t)(nrows * N));
    if (!Ad || !Bd || !tmp) return 1;
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        oracle_decode_nvfp4(A + r * (K / 2), SFA + r * (K / 16), Ad + i * K, 1, K);
    }
    oracle_decode_nvfp4(B, SFB, Bd, N, K);
    contract_f32(Ad, Bd, nrows, N, K, tmp);
    if (C) finish_bf16(tmp, nrows * N, g_a, g_b, 1, C);
    free(Ad);
    free(Bd);
    if (!acc) free(tmp);
    return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
