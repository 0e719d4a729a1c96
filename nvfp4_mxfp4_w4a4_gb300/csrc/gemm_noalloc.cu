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
//   * the counters must be zero when a call starts.  Static device storage
//     is zero when the module loads and every call that finishes without a
//     device timeout leaves the counters zero again; after FP4_ERR_TIMEOUT
//     their contents are unknown.
#include <cuda_runtime.h>

#include <mutex>

#include "fp4lin.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(2) << 20;  // 2 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_gemm_scratch[kScratchBytes];

struct ScratchAddr {
    bool known = false;
    void* ptr = nullptr;
};

ScratchAddr g_addr[kMaxDevices];
std::mutex g_addr_mutex;

// Device address of the array on the current device, looked up once per
// device (the lookup runs with that device current, as the call's own
// launches do).
fp4_status scratch_address(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return FP4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_addr_mutex);
    ScratchAddr& a = g_addr[dev];
    if (!a.known) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_gemm_scratch) != cudaSuccess || p == nullptr)
            return FP4_ERR_CUDA;
        a.ptr = p;
        a.known = true;
    }
    *out = a.ptr;
    return FP4_OK;
}

}  // namespace

extern "C" {

fp4_status fp4_gemm_mxfp4_noalloc(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                                  const void* bias_bf16, void* out_bf16, int64_t M, int64_t N, int64_t K, void* stream)
{
    // the plan depends on the current device's SM count; an unusable device
    // reports 0 here and the call below returns its error
    const size_t need = fp4_gemm_workspace_size(M, N, K);
    if (need > kScratchBytes)
        return FP4_ERR_SHAPE;
    void* scratch = nullptr;
    if (need > 0) {
        const fp4_status st = scratch_address(&scratch);
        if (st != FP4_OK)
            return st;
    }
    return fp4_gemm_mxfp4_ws(a, sa, b, sb, bias_bf16, out_bf16, M, N, K, scratch, scratch ? kScratchBytes : 0,
                             stream);
}

}  // extern "C"
