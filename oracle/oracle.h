/*
 * oracle.h -- plain, slow CPU reference for the W4A4 MXFP4 linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this code; only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * constant generator with the CUDA library.
 *
 * Pages followed (cited by title and section):
 *   [AMD]   "Efficiently Serving NVFP4 Models on AMD Instinct MI350X/MI355X
 *            Accelerators via Online NVFP4 to Quark MXFP4 Requantization"
 *   [OMNI]  "W4A4 MXFP4 Quantization" (vllm-omni user guide, mxfp4.md)
 *   [SGL]   "[SGLang] FP4: 4-bit floating point quantization (NVIDIA NF4)"
 *
 * Every routine works element by element in the order the pages describe,
 * with double precision wherever the pages do not fix a precision.  Scale
 * factors are produced row-major ([rows][K/32]); the swizzled layout the
 * tensor cores read is a separate index function (orc_sf_swizzled_offset).
 *
 * Parity status: every function here is pinned by the CPU tests except the
 * UOS scale rule (orc_mx_shared_exp with alg = 2), which follows one reading
 * of [OMNI] "Single-Scale Block Scaling (OCP / UOS)" and is parity unpinned
 * beyond the two inequalities that reading implies.
 */
#ifndef FP4_ORACLE_H
#define FP4_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- element codecs, from the bit definitions of each format ---------- */
double orc_e2m1_value(unsigned code4);        /* 4-bit code -> value      */
double orc_e4m3_value(unsigned byte);         /* float8_e4m3fn -> value   */
double orc_e8m0_value(unsigned byte);         /* E8M0 -> 2^(b-127) or NaN */
double orc_bf16_value(uint16_t bits);         /* bf16 -> value            */
unsigned orc_e2m1_encode(double q);           /* nearest, ties to even code, saturating, sign copied */
uint16_t orc_bf16_encode(float f);            /* float32 -> bf16, nearest, ties to even */
unsigned orc_e4m3_encode(float t);            /* t >= 0: nearest finite, ties to even code, saturating at 448 */

/* ---- MX shared exponent ([OMNI] Single-Scale Block Scaling) ----------- */
#define ORC_SCALE_OCP 0
#define ORC_SCALE_UOS 2
int orc_mx_shared_exp(double amax, int alg);  /* clamped to [-127, 127]   */

/* One 32-element block -> 16 packed bytes + one E8M0 byte. */
void orc_mx_quantize_block(const float v[32], int alg, uint8_t packed[16], uint8_t* sf);

/* ---- the three hot-path computations (row-major scale output) --------- */
/* NVFP4 decode: v = fp32((E2M1(c) * E4M3(s)) * g)  ([SGL] sections 3-4). */
void orc_nvfp4_dequant(const uint8_t* w_packed, const uint8_t* w_scale, float g,
                       int64_t rows, int64_t K, float* out);
/* NVFP4 -> MXFP4 requantization ([AMD] online requantization pipeline).   */
void orc_requant(const uint8_t* w_packed, const uint8_t* w_scale, float g,
                 int64_t row0, int64_t row1, int64_t K, int alg,
                 uint8_t* out_packed, uint8_t* out_sf);
/* The same with each decoded value rounded to bf16 before the block rule. */
void orc_requant_bf16(const uint8_t* w_packed, const uint8_t* w_scale, float g,
                      int64_t row0, int64_t row1, int64_t K, int alg,
                      uint8_t* out_packed, uint8_t* out_sf);
/* Dynamic MXFP4 quantization of bf16 activations ([AMD] serve-time path).  */
void orc_act_quant(const uint16_t* x_bf16, int64_t row0, int64_t row1, int64_t K,
                   int alg, uint8_t* out_packed, uint8_t* out_sf);

/* W4A4 GEMM over dequantized MXFP4 operands, float64 accumulation.
 * Computes ref[i][j] = sum_k A[rows[i]][k] * B[cols[j]][k] + bias[cols[j]]
 * and absum[i][j] = sum_k |A*B| for the listed rows and columns. bias may be
 * NULL.  sa / sb are row-major E8M0 ([rows][K/32]).                          */
void orc_gemm(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
              const uint16_t* bias_bf16, int64_t K,
              const int64_t* rows, int64_t n_rows, const int64_t* cols, int64_t n_cols,
              double* ref, double* absum);

/* ---- Smooth pre-scale ([OMNI] Pre-Quantized Single-Scale Weights) ------ */
/* mul_scale float32 [K] -> bf16 [K]; returns the count of rejected values
 * (NaN, Inf, <= 0, or overflow / underflow to zero in bf16).               */
int64_t orc_smooth_prepare(const float* mul_scale, int64_t K, uint16_t* out_bf16);
/* out = bf16(x * m) per element (m per input channel, bf16).               */
void orc_smooth_apply(const uint16_t* x_bf16, const uint16_t* m_bf16, int64_t rows, int64_t K,
                      uint16_t* out_bf16);

/* ---- W4A8 fallback ([OMNI] W4A8 fallback, Single-Scale Block Scaling) --- */
/* OCP MX exponent for float8_e4m3fn elements: floor(log2 amax) - 8, clamped. */
int orc_mx8_shared_exp(double amax);
/* One 32-element block -> 32 E4M3 bytes + one E8M0 byte. */
void orc_mx8_quantize_block(const float v[32], uint8_t codes[32], uint8_t* sf);
/* bf16 activations -> MXFP8: codes [rows][K] bytes, row-major E8M0 [rows][K/32]. */
void orc_act_quant_mxfp8(const uint16_t* x_bf16, int64_t row0, int64_t row1, int64_t K,
                         uint8_t* out_codes, uint8_t* out_sf);
/* MXFP8 activations x MXFP4 weights, float64 accumulation; as orc_gemm with
 * a8 [rows][K] E4M3 bytes and sa row-major [rows][K/32].                    */
void orc_gemm_w4a8(const uint8_t* a8, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                   const uint16_t* bias_bf16, int64_t K,
                   const int64_t* rows, int64_t n_rows, const int64_t* cols, int64_t n_cols,
                   double* ref, double* absum);

/* NVFP4 x NVFP4 GEMM ([SGL] sections 5-6): E2M1 codes with row-major E4M3
 * scales per 16 elements (sa [rows][K/16], sb [cols][K/16]), one per-tensor
 * factor alpha (= g_a * g_b), float64 accumulation:
 *   ref[i][j] = alpha * sum_k (c s)_A[rows[i]][k] * (c s)_B[cols[j]][k] + bias
 *   absum[i][j] = |alpha| * sum_k |(c s)_A * (c s)_B|.  bias may be NULL.   */
void orc_gemm_nvfp4(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                    double alpha, const uint16_t* bias_bf16, int64_t K,
                    const int64_t* rows, int64_t n_rows, const int64_t* cols, int64_t n_cols,
                    double* ref, double* absum);

/* ---- DualScale weights ([OMNI] "mxfp4_dualscale"): E2M1 codes [rows][K/2],
 * fine E8M0 [rows][K/32], coarse float32 [rows][K/512]; K % 512 == 0.     */
void orc_dual_dequant(const uint8_t* packed, const uint8_t* fine, const float* coarse, int64_t rows, int64_t K,
                      double* out);
/* bf16 weight -> DualScale (online dual-level quantization, stated reading). */
void orc_dual_quantize(const uint16_t* w_bf16, int64_t row0, int64_t row1, int64_t K, uint8_t* out_packed,
                       uint8_t* out_fine, float* out_coarse);
/* MXFP4 activations x DualScale weights, float64 accumulation (as orc_gemm). */
void orc_gemm_dual(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* fine, const float* coarse,
                   const uint16_t* bias_bf16, int64_t K, const int64_t* rows, int64_t n_rows, const int64_t* cols,
                   int64_t n_cols, double* ref, double* absum);

/* ---- input preparation (NVFP4 producer used to build test inputs) ----- */
float orc_nvfp4_global_scale(const uint16_t* x_bf16, int64_t n);   /* amax/(6*448) */
void orc_nvfp4_quantize(const uint16_t* x_bf16, float g, int64_t row0, int64_t row1,
                        int64_t K, uint8_t* out_packed, uint8_t* out_scale);

/* ---- scale-factor layout the block-scaled MMA reads ------------------- */
int64_t orc_sf_swizzled_bytes(int64_t rows, int64_t kblocks);
int64_t orc_sf_swizzled_offset(int64_t r, int64_t c, int64_t kblocks);
/* Scatter a row-major [rows][kblocks] scale array into the swizzled layout
 * (pad bytes are zero). */
void orc_sf_swizzle(const uint8_t* rowmajor, int64_t rows, int64_t kblocks, uint8_t* out);

#ifdef __cplusplus
}
#endif
#endif
