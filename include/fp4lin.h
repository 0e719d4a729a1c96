/*
 * fp4lin.h -- C ABI of libfp4lin, the W4A4 MXFP4 linear layer on one
 * NVIDIA GB300 (sm_103a).
 *
 * The layer has three parts, all on the GPU:
 *   1. load-time NVFP4 -> MXFP4 weight requantization,
 *   2. dynamic per-batch MXFP4 quantization of bf16 activations,
 *   3. the block-scaled FP4 GEMM over two MXFP4 operands with a bf16
 *      (+ optional bf16 bias) epilogue, dense and grouped (MoE).
 * Beside it: the W4A8 fallback (MXFP8 activations x the same MXFP4
 * weights), the smooth pre-scale x * mul_scale fused into the activation
 * quantizers, and the NVFP4 x NVFP4 GEMM a GPU with native NVFP4 would run
 * without the requantization (the comparison point).
 *
 * Pages that define the operations (cited by title and section):
 *   [AMD]  "Efficiently Serving NVFP4 Models on AMD Instinct MI350X/MI355X
 *           Accelerators via Online NVFP4 to Quark MXFP4 Requantization"
 *   [OMNI] "W4A4 MXFP4 Quantization" (vllm-omni user guide)
 *   [SGL]  "[SGLang] FP4: 4-bit floating point quantization (NVIDIA NF4)"
 *
 * Conventions for every call
 *   - Pointers are DEVICE pointers unless the comment says "host".  The
 *     caller owns every buffer; the library allocates no device memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously; no call synchronizes.
 *   - Argument checks (null pointers, shapes, alignment, device support)
 *     run on the host before any launch and return an error status with
 *     nothing enqueued.  A failed launch returns FP4_ERR_CUDA.
 *   - Device-side waits are bounded.  A wait that gives up records
 *     FP4_ERR_TIMEOUT in a library-owned device status word, which
 *     fp4_get_device_status() reads (that call synchronizes the device).
 *   - Packed FP4 tensors: two E2M1 codes per byte, K-contiguous, element 2j
 *     of a row in the low nibble of byte j, element 2j+1 in the high nibble.
 *   - MXFP4 scale factors are E8M0 bytes (2^(b-127), 0xFF = NaN), one per
 *     32 consecutive K-elements ([OMNI] Overview).  They come in two
 *     layouts:
 *       FP4_SF_ROWMAJOR  [rows][K/32] bytes, as checkpoints store them
 *                        ([OMNI] "Pre-Quantized Single-Scale Weights").
 *       FP4_SF_SWIZZLED  the layout the block-scaled tensor-core MMA reads:
 *                        rows padded to 128, K/32 padded to 4; byte of
 *                        (row r, block c) at
 *                        ((r/128)*ceil(Kb/4) + c/4)*512 + (r%32)*16
 *                          + ((r%128)/32)*4 + c%4,      Kb = K/32.
 *                        Pad bytes are written as 0.
 *     fp4_sf_bytes() gives the size of either layout.
 */
#ifndef FP4LIN_H
#define FP4LIN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FP4LIN_API __attribute__((visibility("default")))
#else
#define FP4LIN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP4_OK = 0,
    FP4_ERR_INVALID_ARG = 1,   /* null pointer, bad enum value            */
    FP4_ERR_SHAPE = 2,         /* dimension not allowed for this call     */
    FP4_ERR_ALIGNMENT = 3,     /* pointer not aligned as required         */
    FP4_ERR_UNSUPPORTED = 4,   /* device is not compute capability 10.3  */
    FP4_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed    */
    FP4_ERR_TIMEOUT = 6        /* a bounded device wait expired           */
} fp4_status;

/* Block scaling rule ([OMNI] "Single-Scale Block Scaling (OCP / UOS)",
 * same numbering as the page's mxfp4_scale_alg setting).
 *   OCP: shared exponent e = floor(log2(amax)) - 2.
 *   UOS: e = the smallest integer with amax <= 7.25 * 2^e; elements still
 *        saturate at 6.  (The page gives only the 7.25 boundary; this is
 *        the reading the library implements.)                              */
typedef enum { FP4_SCALE_OCP = 0, FP4_SCALE_UOS = 2 } fp4_scale_alg;

typedef enum { FP4_SF_SWIZZLED = 0, FP4_SF_ROWMAJOR = 1 } fp4_sf_layout;

/* Quantizer flags.
 *   FP4_QUANT_BF16_INTERMEDIATE  requantization only: round every decoded
 *        NVFP4 value to bf16 (nearest, ties to even) before the MX block
 *        rule, as an implementation that stages the dequantized weight in
 *        bf16 would.  The pages do not say which precision their
 *        dequantized intermediate has; the default is float32.  For bf16
 *        inputs (the activation quantizers) the flag changes nothing.      */
#define FP4_QUANT_BF16_INTERMEDIATE 1u

/* Options for the quantizers.  A NULL pointer means {OCP, SWIZZLED, 0}.
 * Unknown flag bits are rejected with FP4_ERR_INVALID_ARG.                */
typedef struct {
    int32_t scale_alg;   /* fp4_scale_alg */
    int32_t sf_layout;   /* fp4_sf_layout */
    uint32_t flags;      /* FP4_QUANT_* bits */
} fp4_quant_opts;

/* ------------------------------------------------------------------ sizes */

/* Bytes of an E8M0 scale array for `rows` x K elements in the given layout
 * (K must be a multiple of 32; returns 0 otherwise).                      */
FP4LIN_API size_t fp4_sf_bytes(int64_t rows, int64_t K, int32_t sf_layout);

/* Upper bound on the swizzled scale bytes of a grouped activation tensor
 * of total_M rows split into E groups (each group padded to 128 rows).    */
FP4LIN_API size_t fp4_sf_bytes_grouped(int64_t total_M, int32_t E, int64_t K);

/* Human-readable name of a status code (static string). */
FP4LIN_API const char* fp4_status_string(fp4_status s);

/* Reads and clears the device status word on the current device after a
 * device synchronize.  Returns FP4_OK or FP4_ERR_TIMEOUT (or FP4_ERR_CUDA
 * if the synchronize itself failed).  For tests and diagnostics.           */
FP4LIN_API fp4_status fp4_get_device_status(void);

/* Test hook for the bounded device waits (no counterpart on the pages: it
 * exists so that tests can drive the library's failure path without a GPU
 * fault).  Process-wide, read by each later GEMM call when it is enqueued:
 *   wait_limit_ns          limit of every bounded wait of the GEMM kernels
 *                          (0 restores the default of 1 s; otherwise
 *                          1e3 .. 1e10 ns);
 *   withhold_split_signal  1: in a split-K launch (see fp4_gemm_mxfp4_ws),
 *                          the last CTA does not publish its partial sum, so
 *                          the finishing CTA's bounded wait expires: the call
 *                          completes, its output is wrong, and
 *                          fp4_get_device_status() reports FP4_ERR_TIMEOUT;
 *                          the workspace counters are then left non-zero
 *                          (fp4_gemm_mxfp4_ws callers re-zero them).  0: off.
 * Returns FP4_ERR_INVALID_ARG for other values.  Not for production use.    */
FP4LIN_API fp4_status fp4_debug_set_wait_fault(uint64_t wait_limit_ns, int32_t withhold_split_signal);

/* ------------------------------------------------------- requantization */

/* NVFP4 -> MXFP4 weight requantization ([AMD] online requantization
 * pipeline: run once per layer at load; the dequantized intermediate never
 * leaves registers, the result goes straight into a preallocated
 * destination).  NVFP4 layout per [SGL] sections 3-4.
 *
 *   w_packed      [N, K/2] u8    NVFP4 codes (device)
 *   w_scale_e4m3  [N, K/16] u8   float8_e4m3fn block scales (device)
 *   w_global      f32, by value  per-tensor scale; MULTIPLIES the decoded
 *                                values (a loader holding the divisor form
 *                                passes its reciprocal)
 *   out_packed    [N, K/2] u8    MXFP4 codes (device, caller-allocated)
 *   out_scale     E8M0 bytes     fp4_sf_bytes(N, K, layout) (device)
 *
 * Decoding: v = fp32((E2M1(c) * E4M3(s)) * w_global) (one rounding), then
 * v = bf16(v) when opts->flags has FP4_QUANT_BF16_INTERMEDIATE.
 * Encoding per 32-block: amax, shared exponent by the chosen rule clamped
 * to [-127, 127], codes = nearest E2M1 of v / 2^e with ties to the even
 * code, saturating at +-6, sign always kept (-0 -> 0x8).  A block holding
 * NaN or Inf gets scale byte 0xFF and zero codes.
 * Requires N >= 1, K a positive multiple of 32, 16-byte aligned packed
 * pointers.  Outputs must not overlap inputs.
 * fp4_requant_nvfp4_to_mxfp4 uses {OCP, SWIZZLED}.                        */
FP4LIN_API fp4_status fp4_requant_nvfp4_to_mxfp4(const uint8_t* w_packed, const uint8_t* w_scale_e4m3,
                                      float w_global, uint8_t* out_packed, uint8_t* out_scale,
                                      int64_t N, int64_t K, void* stream);
FP4LIN_API fp4_status fp4_requant_nvfp4_to_mxfp4_ex(const uint8_t* w_packed, const uint8_t* w_scale_e4m3,
                                         float w_global, uint8_t* out_packed, uint8_t* out_scale,
                                         int64_t N, int64_t K, const fp4_quant_opts* opts,
                                         void* stream);

/* The same requantization for E tensors of one shape in one launch (all
 * experts of a MoE layer at load time, [AMD] "Native FP4 matmul": MoE
 * experts on MXFP4), each with its own global scale.
 *   w_packed      [E][N][K/2] u8, w_scale_e4m3 [E][N][K/16] u8 (device)
 *   w_global      [E] f32 (DEVICE array), multiplicative as above
 *   out_packed    [E][N][K/2] u8
 *   out_scale     E consecutive arrays of fp4_sf_bytes(N, K, layout) bytes
 *                 (the per-expert scale layout fp4_gemm_mxfp4_grouped reads)
 * Tensor e is bit-identical to fp4_requant_nvfp4_to_mxfp4_ex on its slices
 * with w_global[e].  Requires 1 <= E <= 4096, N >= 1, K a positive multiple
 * of 128 below 2^29 (else FP4_ERR_SHAPE), 32-byte aligned packed pointers,
 * an 8-byte aligned w_scale_e4m3, a 4-byte aligned out_scale (swizzled) and
 * w_global.                                                                 */
FP4LIN_API fp4_status fp4_requant_nvfp4_to_mxfp4_grouped(const uint8_t* w_packed, const uint8_t* w_scale_e4m3,
                                              const float* w_global, uint8_t* out_packed,
                                              uint8_t* out_scale, int32_t E, int64_t N, int64_t K,
                                              const fp4_quant_opts* opts, void* stream);

/* ------------------------------------------------- activation quantizer */

/* Dynamic MXFP4 quantization of bf16 activations ([AMD] serve-time path:
 * the activation scales are computed for every batch; none are stored or
 * calibrated).  Same block rule as the requantization.
 *   x_bf16     [M, K] bf16 (device, 16-byte aligned)
 *   out_packed [M, K/2] u8; out_scale fp4_sf_bytes(M, K, layout) bytes.
 * Requires M >= 0 (M = 0 is a no-op), K a positive multiple of 32.          */
FP4LIN_API fp4_status fp4_quant_act_mxfp4(const void* x_bf16, uint8_t* out_packed, uint8_t* out_scale,
                               int64_t M, int64_t K, const fp4_quant_opts* opts, void* stream);

/* Grouped variant for MoE: rows [row_offsets[e], row_offsets[e+1]) belong
 * to group e.  Scales are always SWIZZLED; group e's scale rows start at
 * sum_{j<e} ceil(rows_j/128)*128, so every group begins on a 128-row tile.
 *   row_offsets  [E+1] int32 (device), non-decreasing, row_offsets[0] = 0,
 *                row_offsets[E] = total_M.  The kernel clamps every offset
 *                to [0, total_M] (and each end to at least its start), so
 *                offsets that break this rule give wrong groups but no
 *                access outside the buffers.
 *   out_scale    fp4_sf_bytes_grouped(total_M, E, K) bytes (device)
 * Only the scale-row tiles a group uses are written (pad rows as 0).       */
FP4LIN_API fp4_status fp4_quant_act_mxfp4_grouped(const void* x_bf16, const int32_t* row_offsets, int32_t E,
                                       int64_t total_M, int64_t K, uint8_t* out_packed,
                                       uint8_t* out_scale, const fp4_quant_opts* opts,
                                       void* stream);

/* ------------------------------------------------------ smooth pre-scale */

/* The Smooth pre-scale of [OMNI] "Pre-Quantized Single-Scale Weights": both
 * the W4A4 and the W4A8 path quantize x * mul_scale, a per-input-channel
 * float32 tensor converted to the activation dtype (bf16) after loading.
 * fp4_smooth_prepare converts it (round to nearest even) and counts the
 * values loading must reject -- NaN, Inf, non-positive, or overflowing /
 * underflowing to zero in bf16 -- into *bad_count (device int32, written
 * by this call; read it after the stream reaches this point, and reject the
 * tensor when it is not 0).
 *   mul_scale  float32 [K] (device), out_bf16 bf16 [K] (device)
 * Requires K >= 1.                                                         */
FP4LIN_API fp4_status fp4_smooth_prepare(const float* mul_scale, void* out_bf16, int64_t K,
                              int32_t* bad_count, void* stream);

/* fp4_quant_act_mxfp4 / fp4_quant_act_mxfp8 of bf16(x * mul_scale): each
 * element times its channel's bf16 scale, the exact float32 product rounded
 * once to bf16, then the quantizer.  mul_scale_bf16: [K] bf16 (device,
 * 16-byte aligned), as fp4_smooth_prepare writes it.  Otherwise the rules
 * of the plain calls.                                                      */
FP4LIN_API fp4_status fp4_quant_act_mxfp4_smooth(const void* x_bf16, const void* mul_scale_bf16,
                                      uint8_t* out_packed, uint8_t* out_scale, int64_t M,
                                      int64_t K, const fp4_quant_opts* opts, void* stream);
FP4LIN_API fp4_status fp4_quant_act_mxfp8_smooth(const void* x_bf16, const void* mul_scale_bf16,
                                      uint8_t* out_e4m3, uint8_t* out_scale, int64_t M, int64_t K,
                                      int32_t sf_layout, void* stream);

/* ----------------------------------------------------------- NVFP4 producer */

/* bf16 -> NVFP4 with a caller-given global scale g (the NVFP4 quantize
 * step of [SGL] section 6, used to build NVFP4 weights from bf16).  Per
 * 16-element block, in float32, one IEEE operation at a time:
 *   s = E4M3_rne_satfinite(bamax / (6*g)); den = E4M3(s) * g;
 *   code_i = E2M1 nearest of x_i / den (ties to even, saturating),
 * signed-zero codes where den is 0 or NaN.  The usual g is
 * amax(x) / (6 * 448), computed by the caller.
 *   out_packed [M, K/2] u8, out_scale_e4m3 [M, K/16] u8 (row-major).
 * Requires K a positive multiple of 16 and 16-byte aligned pointers.       */
FP4LIN_API fp4_status fp4_quant_nvfp4(const void* x_bf16, float g, uint8_t* out_packed,
                           uint8_t* out_scale_e4m3, int64_t M, int64_t K, void* stream);

/* fp4_quant_nvfp4 with a choice of scale layout: FP4_SF_ROWMAJOR writes
 * [M, K/16] (as fp4_quant_nvfp4), FP4_SF_SWIZZLED writes the layout
 * fp4_gemm_nvfp4 reads (the swizzled layout of this header with 16-element
 * blocks, fp4_sf_bytes_nvfp4(M, K, FP4_SF_SWIZZLED) bytes, pad bytes 0).
 * FP4_ERR_INVALID_ARG for another sf_layout value; otherwise the rules of
 * fp4_quant_nvfp4.                                                         */
FP4LIN_API fp4_status fp4_quant_nvfp4_ex(const void* x_bf16, float g, uint8_t* out_packed,
                              uint8_t* out_scale_e4m3, int64_t M, int64_t K, int32_t sf_layout,
                              void* stream);

/* Bytes of the E4M3 scales of an NVFP4 [rows, K] tensor (one per 16
 * elements): row-major rows * K/16; swizzled ceil(rows/128)*128 *
 * ceil(K/64)*4.  0 for K not a positive multiple of 16 or rows < 0.         */
FP4LIN_API size_t fp4_sf_bytes_nvfp4(int64_t rows, int64_t K, int32_t sf_layout);

/* Scale bytes row-major [rows][kblocks] -> the swizzled layout above, for
 * either format (kblocks = K/32 for MXFP4 E8M0 scales, K/16 for NVFP4 E4M3
 * scales).  The step [SGL] section 5 calls swizzle_blockscale, and what a
 * pre-quantized MXFP4 checkpoint ([OMNI] "Pre-Quantized Single-Scale
 * Weights": row-major (N, K/32) bytes) needs before fp4_gemm_mxfp4.
 *   in_rowmajor  rows * kblocks bytes (device)
 *   out          ceil(rows/128) * ceil(kblocks/4) * 512 bytes (device,
 *                4-byte aligned); every byte is written, pad bytes as 0
 * Requires rows >= 0 (0 is a no-op), kblocks >= 1; in and out must not
 * overlap.                                                                  */
FP4LIN_API fp4_status fp4_sf_swizzle(const uint8_t* in_rowmajor, uint8_t* out, int64_t rows,
                          int64_t kblocks, void* stream);

/* ------------------------------------------------------------------ GEMM */

/* W4A4 GEMM on block-scaled FP4 tensor cores ([AMD] "Native FP4 matmul":
 * both operands MXFP4; [OMNI] Configuration: bf16 output with a bf16
 * per-output-channel bias; [SGL] section 6: bias added to the output):
 *   out[m, n] = bf16_rne( sum_k A[m,k] * B[n,k] + bias[n] )
 * with fp32 accumulation.
 *   a     [M, K/2] u8, sa = SWIZZLED scales of A (fp4_sf_bytes(M, K, 0))
 *   b     [N, K/2] u8, sb = SWIZZLED scales of B (fp4_sf_bytes(N, K, 0))
 *   bias  [N] bf16 or NULL
 *   out   [M, N] bf16, row-major
 * Requires K a positive multiple of 128, N a positive multiple of 8,
 * M >= 0 (M = 0 is a no-op), 16-byte aligned a, b, out, sa, sb.            */
FP4LIN_API fp4_status fp4_gemm_mxfp4(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                          const void* bias_bf16, void* out_bf16, int64_t M, int64_t N, int64_t K,
                          void* stream);

/* Bytes of workspace fp4_gemm_mxfp4_ws uses for an M x N x K problem on
 * the current device: 0 when the problem is not split (see below; also 0
 * when the device is unusable), else one 32-bit counter per SM (256-byte
 * padded) followed by one fp32 partial tile (tile width x 128) per CTA.     */
FP4LIN_API size_t fp4_gemm_workspace_size(int64_t M, int64_t N, int64_t K);

/* fp4_gemm_mxfp4 with caller workspace for split-K (the tile scheduling
 * for decode-sized M that the library's design adds to the pages' GEMM).
 * When M <= 64, K % 256 == 0, the 128-row weight tiles number at most half
 * the SMs, the split saves enough work (with n = K / 512 stages per tile,
 * n (S - 1) / S >= 10) and workspace_bytes >= fp4_gemm_workspace_size(M, N,
 * K), the K stages of every tile are split evenly between S = min(8,
 * SMs / tiles, n) CTAs; the CTA holding a tile's first stages adds the others' fp32
 * partial sums in K order (fixed order: the same result on every run on
 * the same device; results can differ in the last bits from
 * fp4_gemm_mxfp4, within the same tolerance).  Otherwise it runs exactly as
 * fp4_gemm_mxfp4.
 *   workspace  device memory, 256-byte aligned, or NULL; the counter area
 *              (the first 256-byte padded 4 * SM-count bytes) must be zero
 *              before the first call; every call that returns without a
 *              device timeout leaves it zero again.  Calls that use the
 *              same workspace must not overlap in time (same stream, or
 *              ordered by events).  Owned by the caller.
 * Same shape and alignment rules as fp4_gemm_mxfp4.                        */
FP4LIN_API fp4_status fp4_gemm_mxfp4_ws(const uint8_t* a, const uint8_t* sa, const uint8_t* b,
                             const uint8_t* sb, const void* bias_bf16, void* out_bf16,
                             int64_t M, int64_t N, int64_t K, void* workspace,
                             size_t workspace_bytes, void* stream);

/* Flags of fp4_gemm_mxfp4_ex. */
#define FP4_GEMM_WEIGHTS_STATIC 1u

/* fp4_gemm_mxfp4_ws with flags (0 gives fp4_gemm_mxfp4_ws exactly).
 *   FP4_GEMM_WEIGHTS_STATIC  the caller states that b and sb are not written
 *     by the kernel enqueued immediately before this call on `stream`
 *     (typically the activation quantizer of a serving step; the weights
 *     were written by work that has finished).  The library launches its
 *     kernels with programmatic stream serialization, so a GEMM starts while
 *     the previous kernel finishes; with this flag it streams the first
 *     pipeline stages of its weights in that window and waits for the
 *     previous kernel only before reading the activations.  Do not set it
 *     when the previous kernel writes the weights (e.g. the requantization
 *     of the same weights just before the GEMM): the GEMM could read them
 *     before they are written.
 * Other flag bits: FP4_ERR_INVALID_ARG.  Otherwise as fp4_gemm_mxfp4_ws
 * (bit-identical results).                                                  */
FP4LIN_API fp4_status fp4_gemm_mxfp4_ex(const uint8_t* a, const uint8_t* sa, const uint8_t* b,
                             const uint8_t* sb, const void* bias_bf16, void* out_bf16,
                             int64_t M, int64_t N, int64_t K, void* workspace,
                             size_t workspace_bytes, uint32_t flags, void* stream);

/* fp4_gemm_mxfp4_ws for callers that cannot provide device memory (a host
 * program holding no device allocator of its own, or a runtime that must
 * not allocate on its request path).  The pages have no counterpart: it
 * exists because of this library's split-K workspace.  The scratch is a
 * fixed 2 MiB array inside the library's device image (one per device,
 * zero when the library loads); nothing is allocated by this call or by
 * the library for it.
 *   Same arguments, results and rules as fp4_gemm_mxfp4_ws with the
 *   array as workspace (bit-identical outputs).
 *   FP4_ERR_SHAPE also when the problem's split-K plan needs more than
 *   2 MiB (fp4_gemm_workspace_size(M, N, K) > 2 MiB): use
 *   fp4_gemm_mxfp4_ws with a workspace of that size instead.
 *   The first call on a device (and the first after a cudaDeviceReset of
 *   it) looks up the array's device address; make that call before
 *   starting a stream capture.
 *   Calls on one device must not overlap in time (the array is shared by
 *   every caller in the process).  A call that uses the array first clears
 *   its split-K counters on `stream` (a memset of under 1 KB; nothing is
 *   allocated), so a call made after FP4_ERR_TIMEOUT, which can leave the
 *   counters set, starts from a clean state.                                */
FP4LIN_API fp4_status fp4_gemm_mxfp4_noalloc(const uint8_t* a, const uint8_t* sa, const uint8_t* b,
                                  const uint8_t* sb, const void* bias_bf16, void* out_bf16,
                                  int64_t M, int64_t N, int64_t K, void* stream);

/* NVFP4 x NVFP4 GEMM on block-scaled FP4 tensor cores, the path [SGL]
 * sections 5-6 take on hardware with native NVFP4 (the comparison point for
 * the MXFP4 path: no requantization, twice the scale bytes):
 *   out[m, n] = bf16_rne( alpha * sum_k (c s)_A[m,k] * (c s)_B[n,k] + bias[n] )
 * with (c s) = E2M1 code times its 16-element block's E4M3 scale and fp32
 * accumulation.  alpha restores the per-tensor global scales: g_a * g_b for
 * multiplicative scales (section 5 forms 1 / (input_global_scale *
 * weight_global_scale) from divisor-form ones).
 *   a, b   [M, K/2], [N, K/2] u8 E2M1 codes
 *   sa, sb SWIZZLED E4M3 scales (fp4_sf_bytes_nvfp4(rows, K, 0)); the tensor
 *          cores read them as unsigned E4M3: every scale byte must be a
 *          finite, non-negative E4M3 value (sign bit clear, not 0x7F), as
 *          fp4_quant_nvfp4_ex writes for finite inputs and g > 0
 *   bias   [N] bf16 or NULL;  out [M, N] bf16, row-major
 *   workspace, workspace_bytes: split-K scratch as in fp4_gemm_mxfp4_ws
 *          (same plan, same size: fp4_gemm_workspace_size(M, N, K)), or NULL
 * Same shape and alignment rules as fp4_gemm_mxfp4.                        */
FP4LIN_API fp4_status fp4_gemm_nvfp4(const uint8_t* a, const uint8_t* sa, const uint8_t* b,
                          const uint8_t* sb, float alpha, const void* bias_bf16, void* out_bf16,
                          int64_t M, int64_t N, int64_t K, void* workspace,
                          size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------- W4A8 fallback */

/* bf16 -> MXFP8 activations for the W4A8 fallback ([OMNI] "W4A8 fallback at
 * selected layers and denoising steps": MXFP8 activations with the same
 * MXFP4 weights; "Single-Scale Block Scaling": float8_e4m3fn elements, the
 * OCP rule, 32-element blocks along K, rint).  Per block: amax, e =
 * floor(log2 amax) - 8 clamped to [-127, 127] (all-zero: -127), scale byte
 * e + 127; each element the nearest E4M3 value of x / 2^e (ties to even,
 * saturating at +-448, sign kept); a block holding NaN or Inf gets scale
 * byte 0xFF and zero bytes.
 *   out_e4m3   [M, K] bytes (device, 16-byte aligned)
 *   out_scale  E8M0 bytes in sf_layout: fp4_sf_bytes(M, K, sf_layout)
 * Requires M >= 0 (0 is a no-op), K a positive multiple of 32.             */
FP4LIN_API fp4_status fp4_quant_act_mxfp8(const void* x_bf16, uint8_t* out_e4m3, uint8_t* out_scale,
                               int64_t M, int64_t K, int32_t sf_layout, void* stream);

/* W4A8 GEMM: MXFP8 activations x MXFP4 weights on block-scaled tensor cores
 * (tcgen05.mma kind::mxf8f6f4), the mixed FP8/FP4 GEMM of [OMNI] "Hardware
 * Support" (bf16 output, bf16 row bias):
 *   out[m, n] = bf16_rne( sum_k A8[m,k] * B[n,k] + bias[n] )
 * with fp32 accumulation.
 *   a_e4m3  [M, K] E4M3 bytes, sa SWIZZLED E8M0 (fp4_sf_bytes(M, K, 0))
 *   b       [N, K/2] MXFP4 codes (32-byte aligned: the tensor memory
 *           accelerator reads them as 4-bit elements), sb SWIZZLED E8M0
 *   workspace, workspace_bytes: split-K scratch as in fp4_gemm_mxfp4_ws,
 *           sized by fp4_gemm_w4a8_workspace_size (this GEMM's stages cover
 *           half as much K, so its split plan differs), or NULL
 * Same shape rules as fp4_gemm_mxfp4.                                      */
FP4LIN_API fp4_status fp4_gemm_w4a8(const uint8_t* a_e4m3, const uint8_t* sa, const uint8_t* b,
                         const uint8_t* sb, const void* bias_bf16, void* out_bf16, int64_t M,
                         int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                         void* stream);

/* Workspace fp4_gemm_w4a8 uses for split-K on an M x N x K problem on the
 * current device (0: not split, or no usable device).                      */
FP4LIN_API size_t fp4_gemm_w4a8_workspace_size(int64_t M, int64_t N, int64_t K);

/* ----------------------------------------------------------- DualScale */

/* DualScale weights ([OMNI] "mxfp4_dualscale", Offline Mode, checkpoint
 * tensor layout): FP4 codes [N, K/2], a fine E8M0 scale per 32 K-elements
 * and a coarse float32 scale per 512 K-elements (weight_dual_scale
 * [N, K/512]); an element's value is E2M1 x 2^(fine - 127) x coarse.
 * K must be a positive multiple of 512 (the page: DualScale needs complete
 * 512-channel groups); otherwise FP4_ERR_SHAPE.                           */

/* Online dual-level quantization of a bf16 weight ([OMNI] "DualScale Online
 * Mode"; the page only names the operation, so this is the library's
 * reading): per row and 512-element group, coarse = float32(amax / 6) over
 * the group's finite magnitudes (1 if none is above zero), then the OCP MX
 * rule on float32(w / coarse) per 32 elements (fine exponent, nearest E2M1
 * code with ties to even, saturating at 6; a NaN/Inf element makes its
 * 32-element block 0xFF with zero codes).
 *   w_bf16      [N, K] bf16 (16-byte aligned)
 *   out_packed  [N, K/2] codes (8-byte aligned)
 *   out_fine    E8M0: FP4_SF_SWIZZLED (fp4_sf_bytes(N, K, 0), 4-byte
 *               aligned, pad rows written as 0) or FP4_SF_ROWMAJOR [N, K/32]
 *   out_coarse  [N, K/512] float32 (4-byte aligned)                         */
FP4LIN_API fp4_status fp4_quant_dualscale(const void* w_bf16, uint8_t* out_packed, uint8_t* out_fine,
                               float* out_coarse, int64_t N, int64_t K, int32_t sf_layout, void* stream);

/* W4A4 GEMM with DualScale weights: MXFP4 activations (a, SWIZZLED sa) times
 * the DualScale weight (b codes, SWIZZLED fine scales sb, coarse [N, K/512]):
 *   out[m, n] = bf16_rne( sum_j coarse[n, j] * P_j[m, n] + bias[n] ),
 *   P_j = the fp32 block-scaled dot product over the j-th 512 elements of K,
 * each group's partial sum taken from the tensor cores and scaled by its
 * coarse scale before it is added (fp32).  workspace / workspace_bytes:
 * split-K scratch as for fp4_gemm_mxfp4_ws (size fp4_gemm_workspace_size),
 * or NULL.  Shape and alignment rules of fp4_gemm_mxfp4, plus K % 512 == 0
 * and a 4-byte aligned coarse array.                                      */
FP4LIN_API fp4_status fp4_gemm_mxfp4_dualscale(const uint8_t* a, const uint8_t* sa, const uint8_t* b,
                                    const uint8_t* sb, const float* coarse, const void* bias_bf16,
                                    void* out_bf16, int64_t M, int64_t N, int64_t K, void* workspace,
                                    size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------ linear layer */

/* Activation formats of fp4_linear. */
typedef enum { FP4_ACT_MXFP4 = 0, FP4_ACT_MXFP8 = 1 } fp4_act_format;

/* Options of fp4_linear.  A NULL pointer means {MXFP4, OCP, no smooth
 * scale, no flags}. */
typedef struct {
    int32_t act_format;          /* fp4_act_format; MXFP8 is the W4A8 fallback   */
    int32_t scale_alg;           /* MXFP4 activations: OCP or UOS; MXFP8: OCP    */
    const void* mul_scale_bf16;  /* smooth pre-scale [K] bf16 (device), or NULL  */
    uint32_t gemm_flags;         /* FP4_GEMM_WEIGHTS_STATIC, FP4_LINEAR_FUSED_QUANT */
} fp4_linear_opts;

/* fp4_linear flag: for MXFP4 activations and M <= 64, quantize the
 * activations inside the GEMM kernel instead of in a kernel before it
 * ([AMD], last section "Fusing activation quantization + GEMM"): the
 * GEMM's otherwise idle epilogue warps quantize each pipeline stage's bf16
 * token slab into shared memory with the activation quantizer's block
 * arithmetic, so the result is bit-identical to the unfused call; the
 * quantized activations are not written to the workspace.  Other shapes
 * and formats ignore the flag.  Measured on GB300 (14336 x 4096 weight,
 * back-to-back calls): no faster than the two-kernel path at M = 1 and
 * slower at larger M, since every weight-tile CTA quantizes the whole token
 * tile; the two-kernel path already overlaps its quantizer with the GEMM's
 * start (programmatic dependent launch, FP4_GEMM_WEIGHTS_STATIC).          */
#define FP4_LINEAR_FUSED_QUANT 2u

/* Bytes of workspace fp4_linear needs for an M x N x K layer with these
 * options on the current device (0 for M = 0, invalid options or no usable
 * device): the split-K scratch of the GEMM, the quantized activations and
 * their scales.                                                            */
FP4LIN_API size_t fp4_linear_workspace_size(int64_t M, int64_t N, int64_t K,
                                 const fp4_linear_opts* opts);

/* The serve-time linear layer in one call: dynamic quantization of the bf16
 * activations (optionally of x * mul_scale), then the block-scaled GEMM with
 * the prepared MXFP4 weights, bf16 output (+ bf16 bias) -- [AMD]'s serve-time
 * path (activations quantized to MXFP4 per batch), [OMNI] Overview / W4A8
 * fallback / Pre-Quantized Single-Scale Weights (smooth), [SGL] section 6
 * (bias after the GEMM).  Exactly fp4_quant_act_mxfp4[_smooth] (or
 * fp4_quant_act_mxfp8[_smooth]) into the workspace followed by
 * fp4_gemm_mxfp4_ex (or fp4_gemm_w4a8) on the same stream (with
 * FP4_LINEAR_FUSED_QUANT and M <= 64: one GEMM launch that quantizes the
 * activations itself, bit-identical output).
 *   x_bf16     [M, K] bf16; w [N, K/2] MXFP4 codes, sw SWIZZLED E8M0
 *   workspace  device memory, 256-byte aligned, at least
 *              fp4_linear_workspace_size(M, N, K, opts) bytes; its first
 *              bytes are the GEMM's split-K counters: zero them once before
 *              the first call (every call that finishes without a device
 *              timeout leaves them zero); calls sharing a workspace must
 *              not overlap in time.  Owned by the caller.
 * Errors: FP4_ERR_INVALID_ARG also for an invalid option or a workspace
 * smaller than the size above.  Shape rules of fp4_gemm_mxfp4; with MXFP8
 * activations w must be 32-byte aligned.                                   */
FP4LIN_API fp4_status fp4_linear(const void* x_bf16, const uint8_t* w, const uint8_t* sw,
                      const void* bias_bf16, void* out_bf16, int64_t M, int64_t N, int64_t K,
                      void* workspace, size_t workspace_bytes, const fp4_linear_opts* opts,
                      void* stream);

/* The MoE form of fp4_linear: grouped activation quantization (MXFP4, OCP
 * or UOS, rows grouped by expert as row_offsets gives) into the workspace,
 * then the grouped GEMM against the experts' weights -- exactly
 * fp4_quant_act_mxfp4_grouped followed by fp4_gemm_mxfp4_grouped on the same
 * stream ([AMD] "Native FP4 matmul": MoE experts on MXFP4).
 *   workspace  device memory, 256-byte aligned, at least
 *              fp4_linear_grouped_workspace_size(total_M, E, K) bytes
 *   opts       scale rule (sf_layout must be SWIZZLED); NULL = OCP
 * Otherwise the rules of the two calls.                                    */
FP4LIN_API size_t fp4_linear_grouped_workspace_size(int64_t total_M, int32_t E, int64_t K);
FP4LIN_API fp4_status fp4_linear_grouped(const void* x_bf16, const int32_t* row_offsets, int32_t E,
                              int64_t total_M, const uint8_t* w, const uint8_t* sw,
                              const void* bias_bf16, void* out_bf16, int64_t N, int64_t K,
                              void* workspace, size_t workspace_bytes,
                              const fp4_quant_opts* opts, void* stream);

/* Grouped (MoE) W4A4 GEMM ([AMD] "Native FP4 matmul": MoE experts on
 * MXFP4): for every expert e and every row m in [row_offsets[e],
 * row_offsets[e+1]):  out[m, :] = A[m, :] . B_e^T (+ bias_e).
 *   a            [total_M, K/2] u8, rows grouped by expert
 *   sa           grouped SWIZZLED scales as written by
 *                fp4_quant_act_mxfp4_grouped
 *   b            [E][N][K/2] u8; sb: E consecutive SWIZZLED arrays of
 *                fp4_sf_bytes(N, K, 0) bytes each
 *   bias         [E][N] bf16 or NULL
 *   row_offsets  [E+1] int32 (device), the same rule as for
 *                fp4_quant_act_mxfp4_grouped (and the same clamping); the
 *                tile walk is derived on the device, so no host
 *                synchronization is needed
 *   out          [total_M, N] bf16
 * Same shape and alignment rules as fp4_gemm_mxfp4, and 1 <= E <= 1024
 * (FP4_ERR_SHAPE otherwise).  Large problems with E <= 239 run on CTA pairs
 * (256 x 256 tiles of one expert), the rest on single CTAs.                 */
FP4LIN_API fp4_status fp4_gemm_mxfp4_grouped(const uint8_t* a, const uint8_t* sa, const uint8_t* b,
                                  const uint8_t* sb, const void* bias_bf16, void* out_bf16,
                                  const int32_t* row_offsets, int32_t E, int64_t total_M,
                                  int64_t N, int64_t K, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* FP4LIN_H */
