// mma_peak.cu -- issue-rate microbenchmark of tcgen05.mma kind::mxf4 (the
// block-scaled FP4 tensor-core instruction the GEMM uses), to measure the
// dense FP4 peak on this GPU.  One CTA per SM; one thread issues a long
// chain of MMAs from shared memory (zero operands, zero scales) into TMEM and
// times it with the SM clock.  Optionally a tcgen05.cp of scale factors is
// issued before every group of MMAs, as the GEMM main loop does.
//
// Exposed through its own small C entry point (fp4_mma_peak_probe) in a
// separate library, used only by the benchmark.
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"

namespace fp4lin {
namespace {

constexpr int kMaxN = 256;

template <int N>
__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int iters, int mmas_per_group, int with_cp,
                                                          unsigned long long* cycles, unsigned int* status)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* a = smem;                       // 128 rows x 128 B
    uint8_t* b = smem + 16384;               // N rows x 128 B
    uint8_t* sf = smem + 16384 + kMaxN * 128;  // 2 KB of scale chunks
    uint64_t* bar = reinterpret_cast<uint64_t*>(sf + 2048);
    uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
    const int total = 16384 + kMaxN * 128 + 2048;
    for (int i = threadIdx.x; i < total / 4; i += blockDim.x)
        reinterpret_cast<uint32_t*>(smem)[i] = 0u;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const int warp = threadIdx.x >> 5;
    if (warp == 0) {
        tmem_alloc(slot, 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *slot;
    if (threadIdx.x == 0) {
        constexpr uint32_t idesc = idesc_mxf4(128, N);
        const uint32_t a_s = smem_u32(a), b_s = smem_u32(b), sf_s = smem_u32(sf);
        const uint32_t sfa_t = tmem + 256, sfb_t = tmem + 256 + 8;
        // scale columns must hold something defined before the first MMA
        for (int g = 0; g < 2; ++g) {
            tc_cp_32x128b_warpx4(sfa_t + 4 * g, smem_desc(sf_s, 0, 128, 0));
            for (int j = 0; j < N / 128 + (N < 128 ? 1 : 0); ++j)
                tc_cp_32x128b_warpx4(sfb_t + 8 * g + 4 * j, smem_desc(sf_s, 0, 128, 0));
        }
        const long long t0 = clock64();
        for (int it = 0; it < iters; ++it) {
            if (with_cp) {
                tc_cp_32x128b_warpx4(sfa_t + 4 * (it & 1), smem_desc(sf_s + 512, 0, 128, 0));
                tc_cp_32x128b_warpx4(sfb_t + 8 * (it & 1), smem_desc(sf_s + 1024, 0, 128, 0));
            }
            for (int k = 0; k < mmas_per_group; ++k)
                tc_mma_mxf4(tmem, smem_desc(a_s + 32 * (k & 3), 16, 1024, 2), smem_desc(b_s + 32 * (k & 3), 16, 1024, 2),
                            idesc_with_sf_id(idesc, (k & 1) * 2u), sfa_t + 4 * (it & 1), sfb_t + 8 * (it & 1), 1u);
        }
        tc_commit(bar);
        mbar_wait_bounded(bar, 0, status, 1u, 2000000000ull);
        const long long t1 = clock64();
        cycles[blockIdx.x] = static_cast<unsigned long long>(t1 - t0);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace
}  // namespace fp4lin

extern "C" __attribute__((visibility("default"))) int fp4_mma_peak_probe(int n, int iters, int mmas_per_group,
                                                                       int with_cp, int num_ctas,
                                                                       unsigned long long* cycles_dev,
                                                                       unsigned int* status_dev, void* stream)
{
    using namespace fp4lin;
    const size_t smem = 16384 + kMaxN * 128 + 2048 + 64 + 1024;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t err = cudaErrorInvalidValue;
#define FP4_PEAK_CASE(NN)                                                                                         \
    case NN:                                                                                                      \
        err = cudaFuncSetAttribute(mma_peak_kernel<NN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
        if (err == cudaSuccess) {                                                                                 \
            mma_peak_kernel<NN><<<num_ctas, 128, smem, s>>>(iters, mmas_per_group, with_cp, cycles_dev, status_dev); \
            err = cudaGetLastError();                                                                             \
        }                                                                                                         \
        break;
    switch (n) {
        FP4_PEAK_CASE(64)
        FP4_PEAK_CASE(128)
        FP4_PEAK_CASE(256)
    default:
        break;
    }
#undef FP4_PEAK_CASE
    return static_cast<int>(err);
}
