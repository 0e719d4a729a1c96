// gemm_noalloc.cu -- the W4A4 GEMM for callers that have no device memory to
// lend the library.
//
// fp4_gemm_mxfp4_ws wants the caller to provide the split-K workspace.  Some
// callers cannot: a plain C host program that links only this library and
// keeps no device allocator of its own, or a serving runtime whose device
// memory is entirely reserved up front (weights, KV cache) and which must
// not allocate on its request path.  This entry point serves them from a
// fixed array in the library's own device image instead: the array exists
// once per device as soon as the module is loaded, so the call allocates
// nothing, ever.
//
// Limits that follow from sharing one fixed array:
//   * size: kScratchBytes.  A problem whose split-K plan needs more is
//     rejected (FP4_ERR_SHAPE) rather than silently run another way;
//   * one call at a time per device: two calls in flight at once (other
//     streams, other threads) would use the same counters and partial tiles;
//   * the split-K counters must be zero when a call's kernel starts.  A call
//     that splits first clears them on its stream (cudaMemsetAsync of the
//     counter area, less than 1 KB; no allocation), so a call after a device
//     timeout (which can leave counters behind) starts clean as well.
#include <cuda_runtime.h>

#include <mutex>

#include "fp4lin.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(2) << 20;  // 2 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_gemm_scratch[kScratchBytes];

struct ScratchAddr {
    unsigned long long ctx = 0;  // context the address belongs to (0: not looked up)
    void* ptr = nullptr;
};

ScratchAddr g_addr[kMaxDevices];
std::mutex g_addr_mutex;

// Device address of the array on the current device, looked up once per
// device and context (the lookup runs with that device current, as the
// call's own launches do).  A device that was reset has a new context, in
// which the library's module, and so the array, is loaded again, possibly
// at another address: the lookup is then repeated.
fp4_status scratch_address(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return FP4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_addr_mutex);
    ScratchAddr& a = g_addr[dev];
    const unsigned long long ctx = fp4lin::current_context_id();
    if (a.ctx == 0 || a.ctx != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_gemm_scratch) != cudaSuccess || p == nullptr)
            return FP4_ERR_CUDA;
        a.ptr = p;
        a.ctx = fp4lin::current_context_id();  // current now: the lookup initialised it
    }
    *out = a.ptr;
    return FP4_OK;
}

}  // namespace

extern "C" {

fp4_status fp4_gemm_mxfp4_noalloc(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                                  const void* bias_bf16, void* out_bf16, int64_t M, int64_t N, int64_t K, void* stream)
{
    // the same host checks as every GEMM entry point, before any CUDA call
    fp4_status st = static_cast<fp4_status>(fp4lin::gemm_check_args(a, sa, b, sb, bias_bf16, out_bf16, M, N, K, 1));
    if (st != FP4_OK || M == 0)
        return st;
    // the plan depends on the current device's SM count; an unusable device
    // reports 0 here and the call below returns its error
    const size_t need = fp4_gemm_workspace_size(M, N, K);
    if (need > kScratchBytes)
        return FP4_ERR_SHAPE;
    void* scratch = nullptr;
    if (need > 0) {
        st = scratch_address(&scratch);
        if (st != FP4_OK)
            return st;
        // the counters start at zero whatever an earlier call left behind
        if (cudaMemsetAsync(scratch, 0, fp4lin::gemm_workspace_counter_bytes(), static_cast<cudaStream_t>(stream)) !=
            cudaSuccess)
            return FP4_ERR_CUDA;
    }
    return fp4_gemm_mxfp4_ws(a, sa, b, sb, bias_bf16, out_bf16, M, N, K, scratch, scratch ? kScratchBytes : 0,
                             stream);
}

}  // extern "C"
