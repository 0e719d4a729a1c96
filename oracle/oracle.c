/*
 * oracle.c -- plain, slow CPU reference for the W4A4 MXFP4 linear layer.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).  Built with gcc, -O2, no fast
 * math and no floating-point contraction, so every operation below is the
 * IEEE operation it reads as.
 *
 * Page abbreviations used in the citations:
 *   [AMD]  "Efficiently Serving NVFP4 Models on AMD Instinct MI350X/MI355X
 *           Accelerators via Online NVFP4 to Quark MXFP4 Requantization"
 *   [OMNI] "W4A4 MXFP4 Quantization" (vllm-omni user guide)
 *   [SGL]  "[SGLang] FP4: 4-bit floating point quantization (NVIDIA NF4)"
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------
 * Element formats.  The pages name the formats ([OMNI] Overview: FP4 E2M1
 * values packed two per byte, float8_e8m0fnu block scales; [SGL] section 4:
 * float8_e4m3fn group scales) but print no bit tables, so each decoder is
 * the format's own bit definition.
 * --------------------------------------------------------------------- */

/* E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
 * Exponent 0 is subnormal (m * 0.5).  No Inf or NaN.                    */
double orc_e2m1_value(unsigned code4)
{
    unsigned s = (code4 >> 3) & 1u, e = (code4 >> 1) & 3u, m = code4 & 1u;
    double mag;
    if (e == 0)
        mag = 0.5 * (double)m;
    else
        mag = ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
    return s ? -mag : mag;
}

/* float8_e4m3fn: sign bit 7, exponent bits 6..3 (bias 7), mantissa 2..0.
 * Exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no Inf.      */
double orc_e4m3_value(unsigned byte)
{
    unsigned s = (byte >> 7) & 1u, e = (byte >> 3) & 15u, m = byte & 7u;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

/* E8M0: an unsigned power of two 2^(b-127); 0xFF is NaN; no zero.       */
double orc_e8m0_value(unsigned byte)
{
    byte &= 0xFFu;
    if (byte == 0xFFu)
        return NAN;
    return ldexp(1.0, (int)byte - 127);
}

/* bf16: the upper 16 bits of an IEEE binary32.                           */
double orc_bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* float32 -> bf16, round to nearest, ties to even (the upper half of the
 * float32 pattern after rounding); NaN stays NaN (quiet), overflow gives
 * Inf.                                                                    */
uint16_t orc_bf16_encode(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (isnan(f))
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lower = u & 0xFFFFu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;                  /* carries into the exponent as it should */
    return (uint16_t)upper;
}

/* Round to the nearest E2M1 value, ties to the even code, saturating at 6
 * ([OMNI] Single-Scale Block Scaling: round_mode "rint"; the largest finite
 * E2M1 value is 6).  Brute force over the eight magnitudes; the sign bit of
 * q is copied, so -0 encodes as 0x8.                                      */
unsigned orc_e2m1_encode(double q)
{
    double mag = fabs(q);
    unsigned best = 0;
    double best_d = INFINITY;
    if (isnan(q))
        return 0u;
    if (mag > 6.0) {
        /* beyond the largest value every distance is largest-first; decide it
         * directly (a brute-force distance would be absorbed for huge |q|) */
        best = 7;
    } else {
        for (unsigned i = 0; i < 8; ++i) {
            double d = fabs(orc_e2m1_value(i) - mag);
            if (d < best_d || (d == best_d && (i & 1u) == 0 && (best & 1u) == 1)) {
                best = i;
                best_d = d;
            }
        }
    }
    return (signbit(q) ? 8u : 0u) | best;
}

/* Round t to the nearest finite float8_e4m3fn value, ties to the even code,
 * saturating at 448.  Brute force over the 127 finite magnitudes.        */
unsigned orc_e4m3_encode(float t)
{
    double mag = fabs((double)t);
    unsigned best = 0;
    double best_d = INFINITY;
    if (isnan(t))
        return 0x7Fu;
    if (mag > 448.0) {
        best = 0x7Eu;
    } else {
        for (unsigned c = 0; c <= 0x7Eu; ++c) {
            double d = fabs(orc_e4m3_value(c) - mag);
            if (d < best_d || (d == best_d && (c & 1u) == 0 && (best & 1u) == 1)) {
                best = c;
                best_d = d;
            }
        }
    }
    return (signbit(t) ? 0x80u : 0u) | best;
}

/* ------------------------------------------------------------------------
 * MX shared exponent of one 32-element block.
 * [OMNI] "Single-Scale Block Scaling (OCP / UOS)": setting 0 is the OCP MX
 * rule, setting 2 is UOS with Qmax = 7.25, where 7.25 only selects the
 * power-of-two scale and the largest element value stays 6.
 *   OCP: e = floor(log2(amax)) - 2   (2 = exponent of E2M1's largest value)
 *   UOS: e = the smallest integer with amax <= 7.25 * 2^e   (reading)
 * All-zero blocks take the smallest exponent.  E8M0 covers 2^-127..2^127,
 * so e is clamped to [-127, 127].
 * --------------------------------------------------------------------- */
int orc_mx_shared_exp(double amax, int alg)
{
    int e, ex;
    if (amax == 0.0)
        return -127;
    (void)frexp(amax, &ex);           /* amax = f * 2^ex, f in [0.5, 1) */
    if (alg == ORC_SCALE_UOS) {
        e = (ex - 1) - 3;
        while (amax > 7.25 * ldexp(1.0, e))
            ++e;
    } else {
        e = (ex - 1) - 2;
    }
    if (e < -127)
        e = -127;
    if (e > 127)
        e = 127;
    return e;
}

/* One block: amax, shared exponent, then every element divided by 2^e and
 * rounded onto E2M1.  A block holding NaN or Inf gets scale byte 0xFF and
 * zero codes (reading; the pages are silent).  Element 2j goes to the low
 * nibble of byte j, element 2j+1 to the high nibble (reading of the
 * float4_e2m1fn_x2 packing named in [OMNI] Overview).                     */
void orc_mx_quantize_block(const float v[32], int alg, uint8_t packed[16], uint8_t* sf)
{
    double amax = 0.0;
    int nonfinite = 0;
    for (int i = 0; i < 32; ++i) {
        if (!isfinite(v[i]))
            nonfinite = 1;
        else if (fabs((double)v[i]) > amax)
            amax = fabs((double)v[i]);
    }
    if (nonfinite) {
        *sf = 0xFFu;
        memset(packed, 0, 16);
        return;
    }
    int e = orc_mx_shared_exp(amax, alg);
    *sf = (uint8_t)(e + 127);
    double scale = ldexp(1.0, e);
    for (int j = 0; j < 16; ++j) {
        unsigned lo = orc_e2m1_encode((double)v[2 * j] / scale);
        unsigned hi = orc_e2m1_encode((double)v[2 * j + 1] / scale);
        packed[j] = (uint8_t)(lo | (hi << 4));
    }
}

/* ------------------------------------------------------------------------
 * NVFP4 decode ([AMD] introduction: packed E2M1 with an FP8 per-block scale
 * and an FP32 per-tensor scale; [SGL] sections 3-4: weight_packed [N, K/2]
 * uint8, weight_scale [N, K/16] float8_e4m3fn, one float32 global scale).
 * The global scale multiplies (reading).  E2M1 * E4M3 is exact, and so is
 * the product with g in double, so the one rounding is the cast to float. */
void orc_nvfp4_dequant(const uint8_t* w_packed, const uint8_t* w_scale, float g,
                       int64_t rows, int64_t K, float* out)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < K; ++k) {
            uint8_t byte = w_packed[r * (K / 2) + k / 2];
            unsigned c = (k % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
            double s = orc_e4m3_value(w_scale[r * (K / 16) + k / 16]);
            out[r * K + k] = (float)(orc_e2m1_value(c) * s * (double)g);
        }
}

/* NVFP4 -> MXFP4 for rows [row0, row1): decode each 32-element block to
 * float, then quantize it as an MX block ([AMD] pipeline description: the
 * dequantized intermediate is quantized to MXFP4 and written to a
 * preallocated destination).  Scale bytes are row-major [rows][K/32].     */
void orc_requant(const uint8_t* w_packed, const uint8_t* w_scale, float g,
                 int64_t row0, int64_t row1, int64_t K, int alg,
                 uint8_t* out_packed, uint8_t* out_sf)
{
    float* v = (float*)malloc(sizeof(float) * (size_t)K);
    for (int64_t r = row0; r < row1; ++r) {
        orc_nvfp4_dequant(w_packed + r * (K / 2), w_scale + r * (K / 16), g, 1, K, v);
        for (int64_t b = 0; b < K / 32; ++b)
            orc_mx_quantize_block(v + 32 * b, alg, out_packed + r * (K / 2) + 16 * b,
                                  out_sf + r * (K / 32) + b);
    }
    free(v);
}

/* The same requantization with a bf16 dequantized intermediate: every
 * decoded value is rounded to bf16 (nearest, ties to even) before the MX
 * block rule, as an implementation that stages the dequantized layer in
 * bf16 would ([AMD] pipeline description: the precision of the dequantized
 * intermediate is not given; float32 above is the default reading).       */
void orc_requant_bf16(const uint8_t* w_packed, const uint8_t* w_scale, float g,
                      int64_t row0, int64_t row1, int64_t K, int alg,
                      uint8_t* out_packed, uint8_t* out_sf)
{
    float* v = (float*)malloc(sizeof(float) * (size_t)K);
    for (int64_t r = row0; r < row1; ++r) {
        orc_nvfp4_dequant(w_packed + r * (K / 2), w_scale + r * (K / 16), g, 1, K, v);
        for (int64_t k = 0; k < K; ++k)
            v[k] = (float)orc_bf16_value(orc_bf16_encode(v[k]));
        for (int64_t b = 0; b < K / 32; ++b)
            orc_mx_quantize_block(v + 32 * b, alg, out_packed + r * (K / 2) + 16 * b,
                                  out_sf + r * (K / 32) + b);
    }
    free(v);
}

/* Dynamic activation quantization ([AMD]: activations are quantized to
 * MXFP4 per batch, with no stored scales).  bf16 -> float is exact.       */
void orc_act_quant(const uint16_t* x_bf16, int64_t row0, int64_t row1, int64_t K,
                   int alg, uint8_t* out_packed, uint8_t* out_sf)
{
    float v[32];
    for (int64_t r = row0; r < row1; ++r)
        for (int64_t b = 0; b < K / 32; ++b) {
            for (int i = 0; i < 32; ++i)
                v[i] = (float)orc_bf16_value(x_bf16[r * K + 32 * b + i]);
            orc_mx_quantize_block(v, alg, out_packed + r * (K / 2) + 16 * b,
                                  out_sf + r * (K / 32) + b);
        }
}

/* ------------------------------------------------------------------------
 * Smooth pre-scale ([OMNI] "Pre-Quantized Single-Scale Weights"): both the
 * W4A4 and the W4A8 path quantize x * mul_scale, a per-input-channel float32
 * tensor converted to the activation dtype (bf16) after loading; NaN, Inf,
 * non-positive values and values that overflow or underflow to zero in bf16
 * are rejected.  The product is taken in the activation dtype: bf16(x * m)
 * with m the bf16 scale (x * m of two bf16 values is exact in float32, then
 * one rounding to bf16).                                                  */
int64_t orc_smooth_prepare(const float* mul_scale, int64_t K, uint16_t* out_bf16)
{
    int64_t bad = 0;
    for (int64_t k = 0; k < K; ++k) {
        float m = mul_scale[k];
        uint16_t b = orc_bf16_encode(m);
        double v = orc_bf16_value(b);
        out_bf16[k] = b;
        if (!(m > 0.0f) || isinf(m) || isinf(v) || v == 0.0)
            ++bad;
    }
    return bad;
}

void orc_smooth_apply(const uint16_t* x_bf16, const uint16_t* m_bf16, int64_t rows, int64_t K,
                      uint16_t* out_bf16)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < K; ++k) {
            float p = (float)(orc_bf16_value(x_bf16[r * K + k]) * orc_bf16_value(m_bf16[k]));
            out_bf16[r * K + k] = orc_bf16_encode(p);
        }
}

/* ------------------------------------------------------------------------
 * MXFP8 activations for the W4A8 fallback ([OMNI] "W4A8 fallback at
 * selected layers and denoising steps": MXFP8 activations with the same
 * MXFP4 weights; "Single-Scale Block Scaling (OCP / UOS)": the A8 path
 * always quantizes to float8_e4m3fn with the OCP rule, 32-element blocks
 * along K and "rint" rounding).  The OCP MX rule with E4M3 elements, whose
 * largest value is 448 = 1.75 * 2^8:
 *   e = floor(log2(amax)) - 8, clamped to [-127, 127] (all-zero: -127);
 *   element = float8_e4m3fn nearest to v / 2^e, ties to the even code,
 *   saturating at +-448 (reading: finite elements never become NaN), sign
 *   kept (-0 is 0x80).
 * A block holding NaN or Inf gets scale byte 0xFF and zero bytes, as in the
 * MXFP4 rule (reading).                                                    */
int orc_mx8_shared_exp(double amax)
{
    int ex;
    if (amax == 0.0)
        return -127;
    (void)frexp(amax, &ex);           /* amax = f * 2^ex, f in [0.5, 1) */
    int e = (ex - 1) - 8;
    if (e < -127)
        e = -127;
    if (e > 127)
        e = 127;
    return e;
}

void orc_mx8_quantize_block(const float v[32], uint8_t codes[32], uint8_t* sf)
{
    double amax = 0.0;
    int nonfinite = 0;
    for (int i = 0; i < 32; ++i) {
        if (!isfinite(v[i]))
            nonfinite = 1;
        else if (fabs((double)v[i]) > amax)
            amax = fabs((double)v[i]);
    }
    if (nonfinite) {
        *sf = 0xFFu;
        memset(codes, 0, 32);
        return;
    }
    int e = orc_mx8_shared_exp(amax);
    *sf = (uint8_t)(e + 127);
    double scale = ldexp(1.0, e);
    for (int i = 0; i < 32; ++i)
        codes[i] = (uint8_t)orc_e4m3_encode((float)((double)v[i] / scale));
}

void orc_act_quant_mxfp8(const uint16_t* x_bf16, int64_t row0, int64_t row1, int64_t K,
                         uint8_t* out_codes, uint8_t* out_sf)
{
    float v[32];
    for (int64_t r = row0; r < row1; ++r)
        for (int64_t b = 0; b < K / 32; ++b) {
            for (int i = 0; i < 32; ++i)
                v[i] = (float)orc_bf16_value(x_bf16[r * K + 32 * b + i]);
            orc_mx8_quantize_block(v, out_codes + r * K + 32 * b, out_sf + r * (K / 32) + b);
        }
}

/* ------------------------------------------------------------------------
 * W4A4 GEMM ([AMD] "Native FP4 matmul": both operands MXFP4; [OMNI]
 * Configuration: bf16 output with a bf16 per-output-channel bias; [SGL]
 * section 6: the bias is added to the GEMM output).  The definition:
 * out[m][n] = sum_k dq(A)[m][k] * dq(B)[n][k] + bias[n], in double.
 * --------------------------------------------------------------------- */
static void dequant_mx_row(const uint8_t* packed, const uint8_t* sf, int64_t K, double* out)
{
    for (int64_t k = 0; k < K; ++k) {
        uint8_t byte = packed[k / 2];
        unsigned c = (k % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
        out[k] = orc_e2m1_value(c) * orc_e8m0_value(sf[k / 32]);
    }
}

void orc_gemm(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
              const uint16_t* bias_bf16, int64_t K,
              const int64_t* rows, int64_t n_rows, const int64_t* cols, int64_t n_cols,
              double* ref, double* absum)
{
    double* arows = (double*)malloc(sizeof(double) * (size_t)(n_rows * K));
    double* brow = (double*)malloc(sizeof(double) * (size_t)K);
    for (int64_t i = 0; i < n_rows; ++i)
        dequant_mx_row(a + rows[i] * (K / 2), sa + rows[i] * (K / 32), K, arows + i * K);
    for (int64_t j = 0; j < n_cols; ++j) {
        int64_t n = cols[j];
        dequant_mx_row(b + n * (K / 2), sb + n * (K / 32), K, brow);
        double bias = bias_bf16 ? orc_bf16_value(bias_bf16[n]) : 0.0;
        for (int64_t i = 0; i < n_rows; ++i) {
            const double* arow = arows + i * K;
            double s = 0.0, sabs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = arow[k] * brow[k];
                s += p;
                sabs += fabs(p);
            }
            ref[i * n_cols + j] = s + bias;
            absum[i * n_cols + j] = sabs;
        }
    }
    free(brow);
    free(arows);
}

/* ------------------------------------------------------------------------
 * W4A8 GEMM ([OMNI] "Hardware Support": the mixed FP8/FP4 GEMM of the W4A8
 * fallback, bf16 output with a bf16 row bias): MXFP8 activations (one E4M3
 * byte per element, E8M0 per 32) times the MXFP4 weights, in double:
 *   out[m][n] = sum_k dq8(A)[m][k] * dq4(B)[n][k] + bias[n]            */
static void dequant_mx8_row(const uint8_t* codes, const uint8_t* sf, int64_t K, double* out)
{
    for (int64_t k = 0; k < K; ++k)
        out[k] = orc_e4m3_value(codes[k]) * orc_e8m0_value(sf[k / 32]);
}

void orc_gemm_w4a8(const uint8_t* a8, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                   const uint16_t* bias_bf16, int64_t K,
                   const int64_t* rows, int64_t n_rows, const int64_t* cols, int64_t n_cols,
                   double* ref, double* absum)
{
    double* arows = (double*)malloc(sizeof(double) * (size_t)(n_rows * K));
    double* brow = (double*)malloc(sizeof(double) * (size_t)K);
    for (int64_t i = 0; i < n_rows; ++i)
        dequant_mx8_row(a8 + rows[i] * K, sa + rows[i] * (K / 32), K, arows + i * K);
    for (int64_t j = 0; j < n_cols; ++j) {
        int64_t n = cols[j];
        dequant_mx_row(b + n * (K / 2), sb + n * (K / 32), K, brow);
        double bias = bias_bf16 ? orc_bf16_value(bias_bf16[n]) : 0.0;
        for (int64_t i = 0; i < n_rows; ++i) {
            const double* arow = arows + i * K;
            double s = 0.0, sabs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = arow[k] * brow[k];
                s += p;
                sabs += fabs(p);
            }
            ref[i * n_cols + j] = s + bias;
            absum[i * n_cols + j] = sabs;
        }
    }
    free(brow);
    free(arows);
}

/* ------------------------------------------------------------------------
 * NVFP4 x NVFP4 GEMM: the FP4 inference path of [SGL] sections 5-6, which
 * runs the GEMM on NVFP4 operands directly (hardware with native NVFP4).
 * Both operands are E2M1 codes with one E4M3 scale per 16 elements; the
 * GEMM works on the scaled codes and one per-tensor factor alpha restores
 * the two global scales (section 5 forms alpha as 1 / (input_global_scale *
 * weight_global_scale) from divisor-form scales; with the multiplicative
 * global scales used here alpha = g_a * g_b); section 6 adds the bias to the
 * GEMM output.  The definition, in double:
 *   out[m][n] = alpha * sum_k (E2M1(a) E4M3(sa))[m][k] * (E2M1(b) E4M3(sb))[n][k]
 *               + bias[n]
 * Every code-times-scale value is exact in double.                       */
static void scaled_nv_row(const uint8_t* packed, const uint8_t* s, int64_t K, double* out)
{
    for (int64_t k = 0; k < K; ++k) {
        uint8_t byte = packed[k / 2];
        unsigned c = (k % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
        out[k] = orc_e2m1_value(c) * orc_e4m3_value(s[k / 16]);
    }
}

void orc_gemm_nvfp4(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                    double alpha, const uint16_t* bias_bf16, int64_t K,
                    const int64_t* rows, int64_t n_rows, const int64_t* cols, int64_t n_cols,
                    double* ref, double* absum)
{
    double* arows = (double*)malloc(sizeof(double) * (size_t)(n_rows * K));
    double* brow = (double*)malloc(sizeof(double) * (size_t)K);
    for (int64_t i = 0; i < n_rows; ++i)
        scaled_nv_row(a + rows[i] * (K / 2), sa + rows[i] * (K / 16), K, arows + i * K);
    for (int64_t j = 0; j < n_cols; ++j) {
        int64_t n = cols[j];
        scaled_nv_row(b + n * (K / 2), sb + n * (K / 16), K, brow);
        double bias = bias_bf16 ? orc_bf16_value(bias_bf16[n]) : 0.0;
        for (int64_t i = 0; i < n_rows; ++i) {
            const double* arow = arows + i * K;
            double s = 0.0, sabs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = arow[k] * brow[k];
                s += p;
                sabs += fabs(p);
            }
            ref[i * n_cols + j] = alpha * s + bias;
            absum[i * n_cols + j] = fabs(alpha) * sabs;
        }
    }
    free(brow);
    free(arows);
}

/* ------------------------------------------------------------------------
 * NVFP4 producer, used only to build NVFP4 test inputs from bf16 tensors.
 * The recipe: g = amax / (6 * 448); per 16-element block the E4M3 scale is
 * the nearest E4M3 to block_amax / (6 g); each element is x / (scale * g)
 * rounded onto E2M1.  All arithmetic is float32, one IEEE operation at a
 * time, in this order:
 *   d6 = 6 * g;  t = bamax / d6;  s = E4M3(t);  den = value(s) * g;
 *   q = x / den;  code = E2M1(q).
 * A zero or NaN den gives signed-zero codes.  Both maxima propagate NaN
 * (as the MX block amax does): a NaN element makes its block's scale NaN
 * (byte 0x7F) and the tensor's global scale NaN.                          */
float orc_nvfp4_global_scale(const uint16_t* x_bf16, int64_t n)
{
    double amax = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double a = fabs(orc_bf16_value(x_bf16[i]));
        if (a > amax || isnan(a))
            amax = a;
        if (isnan(amax))
            break;
    }
    float six_e4m3max = 6.0f * 448.0f;
    return (float)amax / six_e4m3max;
}

void orc_nvfp4_quantize(const uint16_t* x_bf16, float g, int64_t row0, int64_t row1,
                        int64_t K, uint8_t* out_packed, uint8_t* out_scale)
{
    for (int64_t r = row0; r < row1; ++r)
        for (int64_t b = 0; b < K / 16; ++b) {
            const uint16_t* x = x_bf16 + r * K + 16 * b;
            float bamax = 0.0f;
            for (int i = 0; i < 16; ++i) {
                float a = (float)fabs(orc_bf16_value(x[i]));
                if (a > bamax || isnan(a))
                    bamax = a;
                if (isnan(bamax))
                    break;
            }
            float d6 = 6.0f * g;
            float t = bamax / d6;
            unsigned s = orc_e4m3_encode(t);
            float den = (float)orc_e4m3_value(s) * g;
            out_scale[r * (K / 16) + b] = (uint8_t)s;
            for (int j = 0; j < 8; ++j) {
                unsigned code[2];
                for (int h = 0; h < 2; ++h) {
                    float xv = (float)orc_bf16_value(x[2 * j + h]);
                    if (den == 0.0f || isnan(den))
                        code[h] = signbit(xv) ? 8u : 0u;
                    else
                        code[h] = orc_e2m1_encode((double)(xv / den));
                }
                out_packed[r * (K / 2) + 8 * b + j] = (uint8_t)(code[0] | (code[1] << 4));
            }
        }
}

/* ------------------------------------------------------------------------
 * DualScale weights ([OMNI] "mxfp4_dualscale -- DualScale Offline Mode",
 * "Checkpoint tensor layout": FP4 values, a fine E8M0 block scale per 32
 * K-elements (weight_scale [N][K/32]) and a coarse float32 block scale per
 * 512 K-elements (weight_dual_scale [N][K/512][1])).  Reading: an element's
 * value is  E2M1(code) * 2^(fine - 127) * coarse,  in double (exact: the
 * first two factors are a binary fraction with 2 significant bits, the
 * coarse scale a float).
 * --------------------------------------------------------------------- */
static void dequant_dual_row(const uint8_t* packed, const uint8_t* fine, const float* coarse, int64_t K,
                             double* out)
{
    for (int64_t k = 0; k < K; ++k) {
        uint8_t byte = packed[k / 2];
        unsigned c = (k % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
        out[k] = orc_e2m1_value(c) * orc_e8m0_value(fine[k / 32]) * (double)coarse[k / 512];
    }
}

void orc_dual_dequant(const uint8_t* packed, const uint8_t* fine, const float* coarse, int64_t rows, int64_t K,
                      double* out)
{
    for (int64_t r = 0; r < rows; ++r)
        dequant_dual_row(packed + r * (K / 2), fine + r * (K / 32), coarse + r * (K / 512), K, out + r * K);
}

/* Online dual-level quantization of a bf16 weight ([OMNI] "DualScale Online
 * Mode": both scale levels are computed on the fly from the bf16 weight; the
 * page only names the operation).  Reading, per row and 512-element group:
 *   coarse = float32(amax / 6), amax the group's largest finite magnitude
 *            (coarse = 1 for a group without a nonzero finite element), so
 *            that the group's largest element lands on E2M1's largest value;
 *   y      = float32(w / coarse) for every element;
 * then the single-scale OCP MX block rule on y per 32 elements (fine E8M0
 * exponent, nearest E2M1 value with ties to the even code, saturating at
 * 6).  A NaN or Inf element makes only its own 32-element block 0xFF with
 * zero codes, as in the single-scale rule.  Both divisions are IEEE float32
 * operations.                                                              */
void orc_dual_quantize(const uint16_t* w_bf16, int64_t row0, int64_t row1, int64_t K, uint8_t* out_packed,
                       uint8_t* out_fine, float* out_coarse)
{
    float v[32];
    for (int64_t r = row0; r < row1; ++r)
        for (int64_t g = 0; g < K / 512; ++g) {
            const uint16_t* w = w_bf16 + r * K + 512 * g;
            float amax = 0.0f;
            for (int i = 0; i < 512; ++i) {
                float x = (float)orc_bf16_value(w[i]);
                if (isfinite(x) && fabsf(x) > amax)
                    amax = fabsf(x);
            }
            const float coarse = amax > 0.0f ? amax / 6.0f : 1.0f;
            out_coarse[r * (K / 512) + g] = coarse;
            for (int b = 0; b < 16; ++b) {
                for (int i = 0; i < 32; ++i)
                    v[i] = (float)orc_bf16_value(w[32 * b + i]) / coarse;
                orc_mx_quantize_block(v, ORC_SCALE_OCP, out_packed + r * (K / 2) + (512 * g + 32 * b) / 2,
                                      out_fine + r * (K / 32) + 16 * g + b);
            }
        }
}

/* DualScale GEMM (W4A4 with dual-level weight scales): MXFP4 activations
 * times DualScale weights, float64 accumulation:
 *   ref[i][j] = sum_k dq(A)[rows[i]][k] * dqd(B)[cols[j]][k] + bias[cols[j]]
 *   absum[i][j] = sum_k |dq(A) * dqd(B)|.                                  */
void orc_gemm_dual(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* fine, const float* coarse,
                   const uint16_t* bias_bf16, int64_t K, const int64_t* rows, int64_t n_rows, const int64_t* cols,
                   int64_t n_cols, double* ref, double* absum)
{
    double* arows = (double*)malloc(sizeof(double) * (size_t)(n_rows * K));
    double* brow = (double*)malloc(sizeof(double) * (size_t)K);
    for (int64_t i = 0; i < n_rows; ++i)
        dequant_mx_row(a + rows[i] * (K / 2), sa + rows[i] * (K / 32), K, arows + i * K);
    for (int64_t j = 0; j < n_cols; ++j) {
        int64_t n = cols[j];
        dequant_dual_row(b + n * (K / 2), fine + n * (K / 32), coarse + n * (K / 512), K, brow);
        double bias = bias_bf16 ? orc_bf16_value(bias_bf16[n]) : 0.0;
        for (int64_t i = 0; i < n_rows; ++i) {
            const double* arow = arows + i * K;
            double s = 0.0, sabs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = arow[k] * brow[k];
                s += p;
                sabs += fabs(p);
            }
            ref[i * n_cols + j] = s + bias;
            absum[i * n_cols + j] = sabs;
        }
    }
    free(brow);
    free(arows);
}

/* ------------------------------------------------------------------------
 * Scale-factor layout read by the block-scaled tensor-core MMA (reading;
 * [SGL] section 5 only names a "swizzle_blockscale" step).  Rows are grouped
 * in tiles of 128 and block columns in groups of 4; each (tile, group) is a
 * 512-byte chunk in which row r sits at 16*(r%32) + 4*((r%128)/32) and
 * column c at c%4.  Chunks run along the block columns first.  Row count is
 * padded to 128 and the block-column count to 4.
 * --------------------------------------------------------------------- */
int64_t orc_sf_swizzled_bytes(int64_t rows, int64_t kblocks)
{
    int64_t row_tiles = (rows + 127) / 128;
    int64_t col_groups = (kblocks + 3) / 4;
    return row_tiles * col_groups * 512;
}

int64_t orc_sf_swizzled_offset(int64_t r, int64_t c, int64_t kblocks)
{
    int64_t col_groups = (kblocks + 3) / 4;
    int64_t chunk = (r / 128) * col_groups + c / 4;
    return chunk * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
}

void orc_sf_swizzle(const uint8_t* rowmajor, int64_t rows, int64_t kblocks, uint8_t* out)
{
    memset(out, 0, (size_t)orc_sf_swizzled_bytes(rows, kblocks));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < kblocks; ++c)
            out[orc_sf_swizzled_offset(r, c, kblocks)] = rowmajor[r * kblocks + c];
}
