// api.cu -- the extern "C" boundary of libfp4lin.  Validates arguments on
// the host, then enqueues the kernels on the caller's stream.  No call
// allocates device memory and none synchronizes (except
// fp4_get_device_status, which exists to read the device status word).
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "../../include/fp4lin.h"
#include "internal.h"

namespace fp4lin {

unsigned long long current_context_id()
{
    typedef CUresult (*GetCurrentFn)(CUcontext*);
    typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(f);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(f);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

}  // namespace fp4lin

namespace {

// Library-owned device status word: kernels OR flags into it when a
// bounded wait gives up.  One copy per device that loads the library.
__device__ unsigned int g_fp4_device_status;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool checked = false;
    bool supported = false;
    unsigned long long ctx = 0;  // context the status-word address belongs to
    unsigned int* status = nullptr;
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

// Test hooks (fp4_debug_set_wait_fault): the limit of every bounded device
// wait of the GEMMs, and whether one split-K partial withholds its signal.
std::atomic<unsigned long long> g_wait_limit_ns{fp4lin::kWaitLimitNs};
std::atomic<int> g_withhold_split_signal{0};

// Resolves the current device's support and status-word address (once per
// device and context: a reset device gets a new context and a new address).
fp4_status current_device(unsigned int** status)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return FP4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo& d = g_dev[dev];
    if (d.checked && d.supported && d.ctx != fp4lin::current_context_id())
        d.checked = false;
    if (!d.checked) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return FP4_ERR_CUDA;
        // The kernels are built for sm_103a only.
        d.supported = (major == 10 && minor == 3);
        if (d.supported) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_fp4_device_status) != cudaSuccess)
                return FP4_ERR_CUDA;
            d.status = static_cast<unsigned int*>(p);
            d.ctx = fp4lin::current_context_id();  // current now: the lookup initialised it
        }
        d.checked = true;
    }
    if (!d.supported)
        return FP4_ERR_UNSUPPORTED;
    if (status)
        *status = d.status;
    return FP4_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline fp4_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FP4_OK : FP4_ERR_CUDA; }

fp4_status check_opts(const fp4_quant_opts* opts, int* alg, int* swizzled, int* bf16 = nullptr)
{
    *alg = FP4_SCALE_OCP;
    *swizzled = 1;
    if (bf16)
        *bf16 = 0;
    if (!opts)
        return FP4_OK;
    if (opts->scale_alg != FP4_SCALE_OCP && opts->scale_alg != FP4_SCALE_UOS)
        return FP4_ERR_INVALID_ARG;
    if (opts->sf_layout != FP4_SF_SWIZZLED && opts->sf_layout != FP4_SF_ROWMAJOR)
        return FP4_ERR_INVALID_ARG;
    if (opts->flags & ~FP4_QUANT_BF16_INTERMEDIATE)
        return FP4_ERR_INVALID_ARG;
    *alg = opts->scale_alg;
    *swizzled = opts->sf_layout == FP4_SF_SWIZZLED ? 1 : 0;
    if (bf16)
        *bf16 = (opts->flags & FP4_QUANT_BF16_INTERMEDIATE) ? 1 : 0;
    return FP4_OK;
}

constexpr int64_t kMaxDim = int64_t(1) << 31;

}  // namespace

extern "C" {

size_t fp4_sf_bytes(int64_t rows, int64_t K, int32_t sf_layout)
{
    if (rows < 0 || K <= 0 || K % 32 != 0)
        return 0;
    const int64_t kb = K / 32;
    if (sf_layout == FP4_SF_ROWMAJOR)
        return static_cast<size_t>(rows * kb);
    return static_cast<size_t>(((rows + 127) / 128) * 128 * ((kb + 3) / 4) * 4);
}

size_t fp4_sf_bytes_nvfp4(int64_t rows, int64_t K, int32_t sf_layout)
{
    if (rows < 0 || K <= 0 || K % 16 != 0)
        return 0;
    const int64_t kb = K / 16;
    if (sf_layout == FP4_SF_ROWMAJOR)
        return static_cast<size_t>(rows * kb);
    return static_cast<size_t>(((rows + 127) / 128) * 128 * ((kb + 3) / 4) * 4);
}

size_t fp4_sf_bytes_grouped(int64_t total_M, int32_t E, int64_t K)
{
    if (total_M < 0 || E <= 0 || K <= 0 || K % 32 != 0)
        return 0;
    const int64_t tiles = (total_M + static_cast<int64_t>(E) * 127) / 128;
    return static_cast<size_t>(tiles * 128 * ((K / 32 + 3) / 4) * 4);
}

const char* fp4_status_string(fp4_status s)
{
    switch (s) {
    case FP4_OK: return "FP4_OK";
    case FP4_ERR_INVALID_ARG: return "FP4_ERR_INVALID_ARG: null pointer or invalid option";
    case FP4_ERR_SHAPE: return "FP4_ERR_SHAPE: dimension not supported by this call";
    case FP4_ERR_ALIGNMENT: return "FP4_ERR_ALIGNMENT: pointer not 16-byte aligned";
    case FP4_ERR_UNSUPPORTED: return "FP4_ERR_UNSUPPORTED: device is not sm_103";
    case FP4_ERR_CUDA: return "FP4_ERR_CUDA: CUDA runtime call or launch failed";
    case FP4_ERR_TIMEOUT: return "FP4_ERR_TIMEOUT: a bounded device wait expired";
    }
    return "FP4_ERR_UNKNOWN";
}

fp4_status fp4_get_device_status(void)
{
    unsigned int* status = nullptr;
    fp4_status st = current_device(&status);
    if (st != FP4_OK)
        return st;
    if (cudaDeviceSynchronize() != cudaSuccess)
        return FP4_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_fp4_device_status, sizeof v) != cudaSuccess)
        return FP4_ERR_CUDA;
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_fp4_device_status, &zero, sizeof zero) != cudaSuccess)
        return FP4_ERR_CUDA;
    return (v & fp4lin::kStatusTimeout) ? FP4_ERR_TIMEOUT : FP4_OK;
}

fp4_status fp4_debug_set_wait_fault(uint64_t wait_limit_ns, int32_t withhold_split_signal)
{
    if (wait_limit_ns != 0 && (wait_limit_ns < 1000u || wait_limit_ns > 10000000000ull))
        return FP4_ERR_INVALID_ARG;
    if (withhold_split_signal != 0 && withhold_split_signal != 1)
        return FP4_ERR_INVALID_ARG;
    g_wait_limit_ns.store(wait_limit_ns ? wait_limit_ns : fp4lin::kWaitLimitNs);
    g_withhold_split_signal.store(withhold_split_signal);
    return FP4_OK;
}

fp4_status fp4_requant_nvfp4_to_mxfp4_ex(const uint8_t* w_packed, const uint8_t* w_scale_e4m3, float w_global,
                                         uint8_t* out_packed, uint8_t* out_scale, int64_t N, int64_t K,
                                         const fp4_quant_opts* opts, void* stream)
{
    int alg, swz, bf16;
    fp4_status st = check_opts(opts, &alg, &swz, &bf16);
    if (st != FP4_OK)
        return st;
    if (!w_packed || !w_scale_e4m3 || !out_packed || !out_scale)
        return FP4_ERR_INVALID_ARG;
    if (N <= 0 || K <= 0 || K % 32 != 0 || N >= kMaxDim || K >= kMaxDim)
        return FP4_ERR_SHAPE;
    if (!aligned16(w_packed) || !aligned16(out_packed) || (reinterpret_cast<uintptr_t>(w_scale_e4m3) & 1u) ||
        (swz && (reinterpret_cast<uintptr_t>(out_scale) & 3u)))
        return FP4_ERR_ALIGNMENT;
    if ((st = current_device(nullptr)) != FP4_OK)
        return st;
    return from_cuda(fp4lin::launch_requant(w_packed, w_scale_e4m3, w_global, out_packed, out_scale, N, K, alg, swz,
                                            bf16, static_cast<cudaStream_t>(stream)));
}

fp4_status fp4_requant_nvfp4_to_mxfp4(const uint8_t* w_packed, const uint8_t* w_scale_e4m3, float w_global,
                                      uint8_t* out_packed, uint8_t* out_scale, int64_t N, int64_t K, void* stream)
{
    return fp4_requant_nvfp4_to_mxfp4_ex(w_packed, w_scale_e4m3, w_global, out_packed, out_scale, N, K, nullptr,
                                         stream);
}

fp4_status fp4_requant_nvfp4_to_mxfp4_grouped(const uint8_t* w_packed, const uint8_t* w_scale_e4m3,
                                              const float* w_global, uint8_t* out_packed, uint8_t* out_scale,
                                              int32_t E, int64_t N, int64_t K, const fp4_quant_opts* opts,
                                              void* stream)
{
    int alg, swz, bf16;
    fp4_status st = check_opts(opts, &alg, &swz, &bf16);
    if (st != FP4_OK)
        return st;
    if (!w_packed || !w_scale_e4m3 || !w_global || !out_packed || !out_scale)
        return FP4_ERR_INVALID_ARG;
    if (E <= 0 || E > 4096 || N <= 0 || K <= 0 || K % 128 != 0 || N >= kMaxDim || K >= (int64_t(1) << 29) ||
        static_cast<int64_t>(E) * N >= kMaxDim)
        return FP4_ERR_SHAPE;
    if (!fp4lin::requant_flat_ok(w_packed, w_scale_e4m3, out_packed, out_scale, K, swz) ||
        (reinterpret_cast<uintptr_t>(w_global) & 3u))
        return FP4_ERR_ALIGNMENT;
    if ((st = current_device(nullptr)) != FP4_OK)
        return st;
    return from_cuda(fp4lin::launch_requant_grouped(w_packed, w_scale_e4m3, w_global, out_packed, out_scale, E, N, K,
                                                    alg, swz, bf16, static_cast<cudaStream_t>(stream)));
}

static fp4_status act_quant_common(const void* x_bf16, const void* mul, uint8_t* out_packed, uint8_t* out_scale,
                                   int64_t M, int64_t K, const fp4_quant_opts* opts, void* stream)
{
    int alg, swz;
    fp4_status st = check_opts(opts, &alg, &swz);
    if (st != FP4_OK)
        return st;
    if (M < 0 || K <= 0 || K % 32 != 0 || M >= kMaxDim || K >= kMaxDim)
        return FP4_ERR_SHAPE;
    if (M == 0)
        return FP4_OK;
    if (!x_bf16 || !out_packed || !out_scale)
        return FP4_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(out_packed) || (swz && (reinterpret_cast<uintptr_t>(out_scale) & 3u)) ||
        (mul && !aligned16(mul)))
        return FP4_ERR_ALIGNMENT;
    if ((st = current_device(nullptr)) != FP4_OK)
        return st;
    return from_cuda(fp4lin::launch_act_quant(x_bf16, out_packed, out_scale, M, K, alg, swz,
                                              static_cast<cudaStream_t>(stream), mul));
}

fp4_status fp4_quant_act_mxfp4(const void* x_bf16, uint8_t* out_packed, uint8_t* out_scale, int64_t M, int64_t K,
                               const fp4_quant_opts* opts, void* stream)
{
    return act_quant_common(x_bf16, nullptr, out_packed, out_scale, M, K, opts, stream);
}

fp4_status fp4_quant_act_mxfp4_smooth(const void* x_bf16, const void* mul_scale_bf16, uint8_t* out_packed,
                                      uint8_t* out_scale, int64_t M, int64_t K, const fp4_quant_opts* opts,
                                      void* stream)
{
    if (!mul_scale_bf16 && M > 0)
        return FP4_ERR_INVALID_ARG;
    return act_quant_common(x_bf16, mul_scale_bf16, out_packed, out_scale, M, K, opts, stream);
}

fp4_status fp4_quant_act_mxfp4_grouped(const void* x_bf16, const int32_t* row_offsets, int32_t E, int64_t total_M,
                                       int64_t K, uint8_t* out_packed, uint8_t* out_scale,
                                       const fp4_quant_opts* opts, void* stream)
{
    int alg, swz;
    fp4_status st = check_opts(opts, &alg, &swz);
    if (st != FP4_OK)
        return st;
    if (opts && !swz)
        return FP4_ERR_INVALID_ARG;  // grouped scales are always swizzled
    if (E <= 0 || E > 4096 || total_M < 0 || K <= 0 || K % 32 != 0 || total_M >= kMaxDim || K >= kMaxDim)
        return FP4_ERR_SHAPE;
    if (total_M == 0)
        return FP4_OK;
    if (!x_bf16 || !row_offsets || !out_packed || !out_scale)
        return FP4_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(out_packed) || (reinterpret_cast<uintptr_t>(out_scale) & 3u) ||
        (reinterpret_cast<uintptr_t>(row_offsets) & 3u))
        return FP4_ERR_ALIGNMENT;
    if ((st = current_device(nullptr)) != FP4_OK)
        return st;
    return from_cuda(fp4lin::launch_act_quant_grouped(x_bf16, row_offsets, E, total_M, K, out_packed, out_scale, alg,
                                                      static_cast<cudaStream_t>(stream)));
}

fp4_status fp4_quant_nvfp4_ex(const void* x_bf16, float g, uint8_t* out_packed, uint8_t* out_scale_e4m3, int64_t M,
                              int64_t K, int32_t sf_layout, void* stream)
{
    if (M < 0 || K <= 0 || K % 16 != 0 || M >= kMaxDim || K >= kMaxDim)
        return FP4_ERR_SHAPE;
    if (sf_layout != FP4_SF_SWIZZLED && sf_layout != FP4_SF_ROWMAJOR)
        return FP4_ERR_INVALID_ARG;
    if (M == 0)
        return FP4_OK;
    if (!x_bf16 || !out_packed || !out_scale_e4m3)
        return FP4_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || (reinterpret_cast<uintptr_t>(out_packed) & 3u))
        return FP4_ERR_ALIGNMENT;
    fp4_status st;
    if ((st = current_device(nullptr)) != FP4_OK)
        return st;
    return from_cuda(fp4lin::launch_quant_nvfp4(x_bf16, g, out_packed, out_scale_e4m3, M, K,
                                                sf_layout == FP4_SF_SWIZZLED ? 1 : 0,
                                                static_cast<cudaStream_t>(stream)));
}

fp4_status fp4_quant_nvfp4(const void* x_bf16, float g, uint8_t* out_packed, uint8_t* out_scale_e4m3, int64_t M,
                           int64_t K, void* stream)
{
    return fp4_quant_nvfp4_ex(x_bf16, g, out_packed, out_scale_e4m3, M, K, FP4_SF_ROWMAJOR, stream);
}

fp4_status fp4_sf_swizzle(const uint8_t* in_rowmajor, uint8_t* out, int64_t rows, int64_t kblocks, void* stream)
{
    if (rows < 0 || kblocks <= 0 || rows >= kMaxDim || kblocks >= kMaxDim)
        return FP4_ERR_SHAPE;
    if (rows == 0)
        return FP4_OK;
    if (!in_rowmajor || !out)
        return FP4_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(out) & 3u)
        return FP4_ERR_ALIGNMENT;
    fp4_status st;
    if ((st = current_device(nullptr)) != FP4_OK)
        return st;
    return from_cuda(fp4lin::launch_sf_swizzle(in_rowmajor, out, rows, kblocks, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace fp4lin {

// Host-side checks shared by every GEMM entry point (no CUDA call): shapes,
// null pointers (only when M > 0) and 16-byte alignment.
int gemm_check_args(const void* a, const void* sa, const void* b, const void* sb, const void* bias, const void* out,
                    int64_t M, int64_t N, int64_t K, int32_t E)
{
    if (M < 0 || N <= 0 || K <= 0 || K % 128 != 0 || N % 8 != 0 || M >= kMaxDim || N >= kMaxDim || K >= kMaxDim)
        return FP4_ERR_SHAPE;
    if (static_cast<int64_t>(E) * N >= kMaxDim)
        return FP4_ERR_SHAPE;
    if (M == 0)
        return FP4_OK;
    if (!a || !sa || !b || !sb || !out)
        return FP4_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(sa) || !aligned16(b) || !aligned16(sb) || !aligned16(out) ||
        (bias && !aligned16(bias)))
        return FP4_ERR_ALIGNMENT;
    return FP4_OK;
}

}  // namespace fp4lin

extern "C" {

static fp4_status gemm_common(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                              const void* bias, void* out, const int32_t* offsets, int32_t E, int64_t M, int64_t N,
                              int64_t K, void* workspace, size_t workspace_bytes, void* stream,
                              int fmt = fp4lin::kGemmMx, float alpha = 1.0f, uint32_t flags = 0,
                              const void* fused_x = nullptr, const void* fused_mul = nullptr, int fused_uos = 0)
{
    fp4_status st = static_cast<fp4_status>(fp4lin::gemm_check_args(a, sa, b, sb, bias, out, M, N, K, E));
    if (st != FP4_OK || M == 0)
        return st;
    unsigned int* status = nullptr;
    st = current_device(&status);
    if (st != FP4_OK)
        return st;
    fp4lin::GemmArgs args;
    args.a = a;
    args.sa = sa;
    args.b = b;
    args.sb = sb;
    args.bias = bias;
    args.out = out;
    args.row_offsets = offsets;
    args.E = offsets ? E : 1;
    args.M = M;
    args.N = N;
    args.K = K;
    args.status = status;
    args.workspace = workspace;
    args.workspace_bytes = workspace ? workspace_bytes : 0;
    args.fmt = fmt;
    args.alpha = alpha;
    args.early_weights = (flags & FP4_GEMM_WEIGHTS_STATIC) != 0;
    args.x_bf16 = fused_x;
    args.x_mul = fused_mul;
    args.x_uos = fused_uos;
    args.wait_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    args.withhold_split_signal = g_withhold_split_signal.load(std::memory_order_relaxed) != 0;
    return from_cuda(fp4lin::launch_gemm(args, static_cast<cudaStream_t>(stream)));
}

fp4_status fp4_gemm_mxfp4(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                          const void* bias_bf16, void* out_bf16, int64_t M, int64_t N, int64_t K, void* stream)
{
    return gemm_common(a, sa, b, sb, bias_bf16, out_bf16, nullptr, 1, M, N, K, nullptr, 0, stream);
}

size_t fp4_gemm_workspace_size(int64_t M, int64_t N, int64_t K)
{
    if (current_device(nullptr) != FP4_OK)
        return 0;
    return fp4lin::gemm_workspace_bytes(M, N, K, fp4lin::kGemmMx);
}

fp4_status fp4_gemm_mxfp4_ws(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                             const void* bias_bf16, void* out_bf16, int64_t M, int64_t N, int64_t K, void* workspace,
                             size_t workspace_bytes, void* stream)
{
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return FP4_ERR_ALIGNMENT;
    return gemm_common(a, sa, b, sb, bias_bf16, out_bf16, nullptr, 1, M, N, K, workspace, workspace_bytes, stream);
}

fp4_status fp4_gemm_nvfp4(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb, float alpha,
                          const void* bias_bf16, void* out_bf16, int64_t M, int64_t N, int64_t K, void* workspace,
                          size_t workspace_bytes, void* stream)
{
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return FP4_ERR_ALIGNMENT;
    return gemm_common(a, sa, b, sb, bias_bf16, out_bf16, nullptr, 1, M, N, K, workspace, workspace_bytes, stream,
                       fp4lin::kGemmNv, alpha);
}

size_t fp4_gemm_w4a8_workspace_size(int64_t M, int64_t N, int64_t K)
{
    if (current_device(nullptr) != FP4_OK)
        return 0;
    return fp4lin::gemm_workspace_bytes(M, N, K, fp4lin::kGemmW4A8);
}

fp4_status fp4_quant_dualscale(const void* w_bf16, uint8_t* out_packed, uint8_t* out_fine, float* out_coarse,
                               int64_t N, int64_t K, int32_t sf_layout, void* stream)
{
    if (N <= 0 || K <= 0 || K % 512 != 0 || N >= kMaxDim || K >= kMaxDim)
        return FP4_ERR_SHAPE;
    if (sf_layout != FP4_SF_SWIZZLED && sf_layout != FP4_SF_ROWMAJOR)
        return FP4_ERR_INVALID_ARG;
    if (!w_bf16 || !out_packed || !out_fine || !out_coarse)
        return FP4_ERR_INVALID_ARG;
    if (!aligned16(w_bf16) || (reinterpret_cast<uintptr_t>(out_packed) & 7u) ||
        (reinterpret_cast<uintptr_t>(out_coarse) & 3u) ||
        (sf_layout == FP4_SF_SWIZZLED && (reinterpret_cast<uintptr_t>(out_fine) & 3u)))
        return FP4_ERR_ALIGNMENT;
    fp4_status st;
    if ((st = current_device(nullptr)) != FP4_OK)
        return st;
    return from_cuda(fp4lin::launch_dual_quant(w_bf16, out_packed, out_fine, out_coarse, N, K,
                                               sf_layout == FP4_SF_SWIZZLED ? 1 : 0,
                                               static_cast<cudaStream_t>(stream)));
}

fp4_status fp4_gemm_mxfp4_dualscale(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                                    const float* coarse, const void* bias_bf16, void* out_bf16, int64_t M, int64_t N,
                                    int64_t K, void* workspace, size_t workspace_bytes, void* stream)
{
    if (K <= 0 || K % 512 != 0)
        return FP4_ERR_SHAPE;
    if (M > 0 && !coarse)
        return FP4_ERR_INVALID_ARG;
    if (coarse && (reinterpret_cast<uintptr_t>(coarse) & 3u))
        return FP4_ERR_ALIGNMENT;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return FP4_ERR_ALIGNMENT;
    fp4_status st = static_cast<fp4_status>(fp4lin::gemm_check_args(a, sa, b, sb, bias_bf16, out_bf16, M, N, K, 1));
    if (st != FP4_OK || M == 0)
        return st;
    unsigned int* status = nullptr;
    if ((st = current_device(&status)) != FP4_OK)
        return st;
    fp4lin::GemmArgs args;
    args.a = a;
    args.sa = sa;
    args.b = b;
    args.sb = sb;
    args.bias = bias_bf16;
    args.out = out_bf16;
    args.row_offsets = nullptr;
    args.E = 1;
    args.M = M;
    args.N = N;
    args.K = K;
    args.status = status;
    args.workspace = workspace;
    args.workspace_bytes = workspace ? workspace_bytes : 0;
    args.fmt = fp4lin::kGemmDual;
    args.coarse = coarse;
    args.wait_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    return from_cuda(fp4lin::launch_gemm(args, static_cast<cudaStream_t>(stream)));
}

fp4_status fp4_gemm_w4a8(const uint8_t* a_e4m3, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                         const void* bias_bf16, void* out_bf16, int64_t M, int64_t N, int64_t K, void* workspace,
                         size_t workspace_bytes, void* stream)
{
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return FP4_ERR_ALIGNMENT;
    if (b && (reinterpret_cast<uintptr_t>(b) & 31u))
        return FP4_ERR_ALIGNMENT;  // the TMA reads the weights as 4-bit elements: 32-byte aligned base
    return gemm_common(a_e4m3, sa, b, sb, bias_bf16, out_bf16, nullptr, 1, M, N, K, workspace, workspace_bytes,
                       stream, fp4lin::kGemmW4A8);
}

static fp4_status act_quant8_common(const void* x_bf16, const void* mul, uint8_t* out_e4m3, uint8_t* out_scale,
                                    int64_t M, int64_t K, int32_t sf_layout, void* stream)
{
    if (M < 0 || K <= 0 || K % 32 != 0 || M >= kMaxDim || K >= kMaxDim)
        return FP4_ERR_SHAPE;
    if (sf_layout != FP4_SF_SWIZZLED && sf_layout != FP4_SF_ROWMAJOR)
        return FP4_ERR_INVALID_ARG;
    if (M == 0)
        return FP4_OK;
    if (!x_bf16 || !out_e4m3 || !out_scale)
        return FP4_ERR_INVALID_ARG;
    const bool swz = sf_layout == FP4_SF_SWIZZLED;
    if (!aligned16(x_bf16) || !aligned16(out_e4m3) || (swz && (reinterpret_cast<uintptr_t>(out_scale) & 3u)) ||
        (mul && !aligned16(mul)))
        return FP4_ERR_ALIGNMENT;
    fp4_status st;
    if ((st = current_device(nullptr)) != FP4_OK)
        return st;
    return from_cuda(fp4lin::launch_act_quant_mxfp8(x_bf16, out_e4m3, out_scale, M, K, swz ? 1 : 0,
                                                    static_cast<cudaStream_t>(stream), mul));
}

fp4_status fp4_quant_act_mxfp8(const void* x_bf16, uint8_t* out_e4m3, uint8_t* out_scale, int64_t M, int64_t K,
                               int32_t sf_layout, void* stream)
{
    return act_quant8_common(x_bf16, nullptr, out_e4m3, out_scale, M, K, sf_layout, stream);
}

fp4_status fp4_quant_act_mxfp8_smooth(const void* x_bf16, const void* mul_scale_bf16, uint8_t* out_e4m3,
                                      uint8_t* out_scale, int64_t M, int64_t K, int32_t sf_layout, void* stream)
{
    if (!mul_scale_bf16 && M > 0)
        return FP4_ERR_INVALID_ARG;
    return act_quant8_common(x_bf16, mul_scale_bf16, out_e4m3, out_scale, M, K, sf_layout, stream);
}

fp4_status fp4_smooth_prepare(const float* mul_scale, void* out_bf16, int64_t K, int32_t* bad_count, void* stream)
{
    if (K <= 0 || K >= kMaxDim)
        return FP4_ERR_SHAPE;
    if (!mul_scale || !out_bf16 || !bad_count)
        return FP4_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(mul_scale) & 3u) || (reinterpret_cast<uintptr_t>(out_bf16) & 1u) ||
        (reinterpret_cast<uintptr_t>(bad_count) & 3u))
        return FP4_ERR_ALIGNMENT;
    fp4_status st;
    if ((st = current_device(nullptr)) != FP4_OK)
        return st;
    return from_cuda(fp4lin::launch_smooth_prepare(mul_scale, out_bf16, K, bad_count,
                                                   static_cast<cudaStream_t>(stream)));
}

fp4_status fp4_gemm_mxfp4_ex(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                             const void* bias_bf16, void* out_bf16, int64_t M, int64_t N, int64_t K, void* workspace,
                             size_t workspace_bytes, uint32_t flags, void* stream)
{
    if (flags & ~static_cast<uint32_t>(FP4_GEMM_WEIGHTS_STATIC))
        return FP4_ERR_INVALID_ARG;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return FP4_ERR_ALIGNMENT;
    return gemm_common(a, sa, b, sb, bias_bf16, out_bf16, nullptr, 1, M, N, K, workspace, workspace_bytes, stream,
                       fp4lin::kGemmMx, 1.0f, flags);
}

// ----------------------------------------------------------- linear layer
namespace {

struct LinearPlan {
    int fmt;          // GemmFormat
    int alg;          // activation scale rule
    size_t split;     // split-K scratch at offset 0
    size_t act_off;   // quantized activations
    size_t sf_off;    // their swizzled scales
    size_t total;
};

inline size_t round256(size_t x) { return (x + 255) / 256 * 256; }

fp4_status linear_plan(int64_t M, int64_t N, int64_t K, const fp4_linear_opts* o, LinearPlan* pl)
{
    if (M < 0 || N <= 0 || K <= 0 || K % 128 != 0 || N % 8 != 0 || M >= kMaxDim || N >= kMaxDim || K >= kMaxDim)
        return FP4_ERR_SHAPE;
    const int act = o ? o->act_format : FP4_ACT_MXFP4;
    const int alg = o ? o->scale_alg : FP4_SCALE_OCP;
    if (act != FP4_ACT_MXFP4 && act != FP4_ACT_MXFP8)
        return FP4_ERR_INVALID_ARG;
    if (alg != FP4_SCALE_OCP && alg != FP4_SCALE_UOS)
        return FP4_ERR_INVALID_ARG;
    if (act == FP4_ACT_MXFP8 && alg != FP4_SCALE_OCP)
        return FP4_ERR_INVALID_ARG;  // the A8 path always takes the OCP rule
    if (o && (o->gemm_flags & ~static_cast<uint32_t>(FP4_GEMM_WEIGHTS_STATIC | FP4_LINEAR_FUSED_QUANT)))
        return FP4_ERR_INVALID_ARG;
    pl->fmt = act == FP4_ACT_MXFP8 ? fp4lin::kGemmW4A8 : fp4lin::kGemmMx;
    pl->alg = alg;
    pl->split = current_device(nullptr) == FP4_OK ? round256(fp4lin::gemm_workspace_bytes(M, N, K, pl->fmt)) : 0;
    pl->act_off = pl->split;
    const size_t act_bytes = static_cast<size_t>(M) * static_cast<size_t>(act == FP4_ACT_MXFP8 ? K : K / 2);
    pl->sf_off = pl->act_off + round256(act_bytes);
    pl->total = pl->sf_off + round256(fp4_sf_bytes(M, K, FP4_SF_SWIZZLED));
    return FP4_OK;
}

}  // namespace

size_t fp4_linear_workspace_size(int64_t M, int64_t N, int64_t K, const fp4_linear_opts* opts)
{
    LinearPlan pl;
    if (M <= 0 || linear_plan(M, N, K, opts, &pl) != FP4_OK)
        return 0;
    return pl.total;
}

fp4_status fp4_linear(const void* x_bf16, const uint8_t* w, const uint8_t* sw, const void* bias_bf16, void* out_bf16,
                      int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                      const fp4_linear_opts* opts, void* stream)
{
    LinearPlan pl;
    fp4_status st = linear_plan(M, N, K, opts, &pl);
    if (st != FP4_OK)
        return st;
    if (M == 0)
        return FP4_OK;
    if (!x_bf16 || !w || !sw || !out_bf16 || !workspace)
        return FP4_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return FP4_ERR_ALIGNMENT;
    if (pl.fmt == fp4lin::kGemmW4A8 && (reinterpret_cast<uintptr_t>(w) & 31u))
        return FP4_ERR_ALIGNMENT;
    if (workspace_bytes < pl.total)
        return FP4_ERR_INVALID_ARG;
    uint8_t* base = static_cast<uint8_t*>(workspace);
    uint8_t* a = base + pl.act_off;
    uint8_t* sa = base + pl.sf_off;
    const void* mul = opts ? opts->mul_scale_bf16 : nullptr;
    const uint32_t gflags = opts ? opts->gemm_flags : 0u;
    if ((gflags & FP4_LINEAR_FUSED_QUANT) && pl.fmt == fp4lin::kGemmMx && M <= 64) {
        // the GEMM quantizes the activations itself (a and sa are not read)
        if (!aligned16(x_bf16) || (mul && !aligned16(mul)))
            return FP4_ERR_ALIGNMENT;
        return gemm_common(a, sa, w, sw, bias_bf16, out_bf16, nullptr, 1, M, N, K, pl.split ? base : nullptr,
                           pl.split, stream, fp4lin::kGemmMx, 1.0f, gflags & FP4_GEMM_WEIGHTS_STATIC, x_bf16, mul,
                           pl.alg == FP4_SCALE_UOS ? 1 : 0);
    }
    if (pl.fmt == fp4lin::kGemmW4A8)
        st = act_quant8_common(x_bf16, mul, a, sa, M, K, FP4_SF_SWIZZLED, stream);
    else {
        const fp4_quant_opts qo = {pl.alg, FP4_SF_SWIZZLED, 0u};
        st = act_quant_common(x_bf16, mul, a, sa, M, K, &qo, stream);
    }
    if (st != FP4_OK)
        return st;
    return gemm_common(a, sa, w, sw, bias_bf16, out_bf16, nullptr, 1, M, N, K, pl.split ? base : nullptr, pl.split,
                       stream, pl.fmt, 1.0f, gflags & FP4_GEMM_WEIGHTS_STATIC);
}

size_t fp4_linear_grouped_workspace_size(int64_t total_M, int32_t E, int64_t K)
{
    if (total_M <= 0 || E <= 0 || K <= 0 || K % 32 != 0)
        return 0;
    return round256(static_cast<size_t>(total_M) * static_cast<size_t>(K / 2)) +
           round256(fp4_sf_bytes_grouped(total_M, E, K));
}

fp4_status fp4_linear_grouped(const void* x_bf16, const int32_t* row_offsets, int32_t E, int64_t total_M,
                              const uint8_t* w, const uint8_t* sw, const void* bias_bf16, void* out_bf16, int64_t N,
                              int64_t K, void* workspace, size_t workspace_bytes, const fp4_quant_opts* opts,
                              void* stream)
{
    int alg, swz;
    fp4_status st = check_opts(opts, &alg, &swz);
    if (st != FP4_OK)
        return st;
    if (opts && !swz)
        return FP4_ERR_INVALID_ARG;
    if (E <= 0 || E > fp4lin::kMaxGroupedExperts || total_M < 0 || N <= 0 || K <= 0 || K % 128 != 0 ||
        N % 8 != 0 || total_M >= kMaxDim || N >= kMaxDim || K >= kMaxDim || static_cast<int64_t>(E) * N >= kMaxDim)
        return FP4_ERR_SHAPE;
    if (total_M == 0)
        return FP4_OK;
    if (!workspace)
        return FP4_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return FP4_ERR_ALIGNMENT;
    if (workspace_bytes < fp4_linear_grouped_workspace_size(total_M, E, K))
        return FP4_ERR_INVALID_ARG;
    uint8_t* a = static_cast<uint8_t*>(workspace);
    uint8_t* sa = a + round256(static_cast<size_t>(total_M) * static_cast<size_t>(K / 2));
    st = fp4_quant_act_mxfp4_grouped(x_bf16, row_offsets, E, total_M, K, a, sa, opts, stream);
    if (st != FP4_OK)
        return st;
    return fp4_gemm_mxfp4_grouped(a, sa, w, sw, bias_bf16, out_bf16, row_offsets, E, total_M, N, K, stream);
}

fp4_status fp4_gemm_mxfp4_grouped(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                                  const void* bias_bf16, void* out_bf16, const int32_t* row_offsets, int32_t E,
                                  int64_t total_M, int64_t N, int64_t K, void* stream)
{
    if (E <= 0 || E > fp4lin::kMaxGroupedExperts)
        return FP4_ERR_SHAPE;
    if (total_M > 0 && !row_offsets)
        return FP4_ERR_INVALID_ARG;
    if (row_offsets && (reinterpret_cast<uintptr_t>(row_offsets) & 3u))
        return FP4_ERR_ALIGNMENT;
    return gemm_common(a, sa, b, sb, bias_bf16, out_bf16, row_offsets, E, total_M, N, K, nullptr, 0, stream);
}

}  // extern "C"
