// internal.h -- host-side launchers shared between the C ABI layer and the
// kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace fp4lin {

// Launches `kern` with programmatic stream serialization allowed, so that
// its prologue overlaps the tail of the previous kernel in the stream (the
// kernel itself waits for that kernel before touching global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// The same for a kernel whose blocks wait on one another (the split-K GEMM:
// a tile's first CTA waits for the others' partial sums): a cooperative
// launch, which the runtime starts only when every block is resident at
// once.  Programmatic serialization is kept where the runtime takes both
// attributes together; otherwise the cooperative launch goes alone.
template <typename... KArgs, typename... Args>
cudaError_t launch_coop(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                        Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t err = cudaLaunchKernelEx(&cfg, kern, args...);
    if (err == cudaSuccess)
        return err;
    (void)cudaGetLastError();  // a refused attribute combination leaves no error behind
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Identifier of the CUDA context current on the calling thread, unique for
// the life of the process (0 when no context is current).  Per-device caches
// of device addresses and function attributes are keyed by it: after a
// cudaDeviceReset the device gets a new context, with the library's module
// loaded again and its attributes unset.
unsigned long long current_context_id();

// Status word bits a kernel sets in the library-owned device status word.
constexpr unsigned int kStatusTimeout = 1u;

// Largest expert count of the grouped GEMM (its tile walk keeps a per-expert
// prefix in shared memory).
constexpr int kMaxGroupedExperts = 1024;

// Upper bound of every bounded device wait (nanoseconds of wall time).
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// alg: 0 OCP, 2 UOS; bf16: round the decoded values to bf16 first.
cudaError_t launch_requant(const uint8_t* wp, const uint8_t* ws, float g, uint8_t* op, uint8_t* osf,
                           int64_t N, int64_t K, int alg, int swizzled, int bf16, cudaStream_t stream);

// E tensors [E][N][K/2] with global scales g_dev[E] (device); needs
// requant_flat_ok (K % 128 == 0, K < 2^29 and aligned arrays).
cudaError_t launch_requant_grouped(const uint8_t* wp, const uint8_t* ws, const float* g_dev, uint8_t* op,
                                   uint8_t* osf, int E, int64_t N, int64_t K, int alg, int swizzled, int bf16,
                                   cudaStream_t stream);

bool requant_flat_ok(const uint8_t* wp, const uint8_t* ws, const uint8_t* op, const uint8_t* osf, int64_t K,
                     int swizzled);

// mul: bf16 [K] smooth pre-scale or null.
cudaError_t launch_act_quant(const void* x, uint8_t* op, uint8_t* osf, int64_t M, int64_t K, int alg,
                             int swizzled, cudaStream_t stream, const void* mul = nullptr);

// bf16 -> MXFP8 (E4M3 codes [M, K], E8M0 per 32, OCP rule) for the W4A8 path.
cudaError_t launch_act_quant_mxfp8(const void* x, uint8_t* op, uint8_t* osf, int64_t M, int64_t K, int swizzled,
                                   cudaStream_t stream, const void* mul = nullptr);

// Smooth pre-scale: float32 [K] -> bf16 [K], *bad = count of rejected values.
cudaError_t launch_smooth_prepare(const float* m, void* out, int64_t K, int32_t* bad, cudaStream_t stream);

cudaError_t launch_act_quant_grouped(const void* x, const int32_t* offsets, int E, int64_t total_M,
                                     int64_t K, uint8_t* op, uint8_t* osf, int alg, cudaStream_t stream);

cudaError_t launch_quant_nvfp4(const void* x, float g, uint8_t* op, uint8_t* osf, int64_t M, int64_t K,
                               int swizzled, cudaStream_t stream);

// Row-major [rows][kb] scale bytes -> swizzled layout (any block size).
cudaError_t launch_sf_swizzle(const uint8_t* in, uint8_t* out, int64_t rows, int64_t kb, cudaStream_t stream);

// bf16 [N, K] -> DualScale (K % 512 == 0): codes [N, K/2], fine E8M0 per 32
// (swizzled or row-major [N, K/32]), coarse float32 [N, K/512].
cudaError_t launch_dual_quant(const void* w, uint8_t* op, uint8_t* ofine, float* ocoarse, int64_t N, int64_t K,
                              int swizzled, cudaStream_t stream);

// Operand formats of the GEMM: both MXFP4; both NVFP4 (E4M3 scales per 16
// elements, alpha); MXFP8 activations (a: [M, K] E4M3 bytes) x MXFP4 weights.
enum GemmFormat : int { kGemmMx = 0, kGemmNv = 1, kGemmW4A8 = 2, kGemmDual = 3 };

// Dense (offsets == nullptr) or grouped GEMM.
struct GemmArgs {
    const uint8_t* a;
    const uint8_t* sa;
    const uint8_t* b;
    const uint8_t* sb;
    const void* bias;
    void* out;
    const int32_t* row_offsets;  // grouped only
    int E;                       // grouped only (1 for dense)
    int64_t M;                   // rows of A (total rows when grouped)
    int64_t N;
    int64_t K;
    unsigned int* status;
    void* workspace;             // split-K scratch (nullptr: none)
    size_t workspace_bytes;
    int fmt = 0;                 // GemmFormat
    float alpha = 1.0f;          // NVFP4: factor on the accumulator before the bias
    const float* coarse = nullptr;  // DualScale: float32 coarse weight scales [N, K/512]
    bool early_weights = false;  // the weights are not written by the preceding kernel in the stream
    unsigned long long wait_ns = kWaitLimitNs;  // limit of every bounded device wait of the launch
    bool withhold_split_signal = false;  // test hook: one split-K partial never signals its finisher
    // M <= 64 MXFP4 only: bf16 activations [M, K] that the GEMM quantizes
    // itself (a and sa unused), with an optional smooth pre-scale and rule
    const void* x_bf16 = nullptr;
    const void* x_mul = nullptr;
    int x_uos = 0;
};

cudaError_t launch_gemm(const GemmArgs& args, cudaStream_t stream);

// MXFP4 GEMM on 256 x 256 output tiles computed by CTA pairs (tcgen05
// cta_group::2), dense or grouped (row_offsets set, E <= gemm_pair_max_experts());
// used by launch_gemm for large problems.
cudaError_t launch_gemm_pair(const GemmArgs& args, cudaStream_t stream);
int gemm_pair_max_experts();

// Host helpers shared by the GEMM translation units (gemm.cu).
// Operand kinds of make_operand_map.
enum : int { kOpFp4Packed = 0, kOpBytes = 1, kOpFp4Expanded = 2 };
bool make_operand_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows, int kc, int kind);
bool make_output_map(CUtensorMap* map, void* base, int64_t rows, int64_t cols, int box_cols, int box_rows,
                     CUtensorMapSwizzle swizzle);
int sm_count();

// Host-side argument checks of the GEMM entry points; returns an fp4_status
// value (FP4_OK = 0), makes no CUDA call.
int gemm_check_args(const void* a, const void* sa, const void* b, const void* sb, const void* bias, const void* out,
                    int64_t M, int64_t N, int64_t K, int32_t E);

// Bytes at the start of a split-K workspace that hold the per-CTA counters
// (zero between calls) on the current device.
size_t gemm_workspace_counter_bytes();

// Workspace the GEMM uses for split-K on this problem on the current device
// (0: the problem is not split): a zero-initialised counter per SM (256-byte
// padded), then one fp32 partial tile per CTA.
size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int fmt);

}  // namespace fp4lin
