// mma_peak.cu -- issue-rate microbenchmark of the block-scaled FP4
// tensor-core instructions, to measure the dense FP4 peak on this GPU and to
// find which form of the instruction is fastest for MXFP4 operands.
//
// Forms (all E2M1 operands, fp32 accumulation in TMEM):
//   kind 0  tcgen05.mma kind::mxf4      scale_vec::2X, UE8M0 scales (block 32)
//   kind 1  tcgen05.mma kind::mxf4nvf4  scale_vec::2X, UE8M0 scales (block 32)
//   kind 2  tcgen05.mma kind::mxf4nvf4  scale_vec::4X, UE8M0 scales (block 16)
//   kind 3  tcgen05.mma kind::mxf4nvf4  scale_vec::4X, UE4M3 scales (block 16, NVFP4)
// and, for the W4A8 path, kind 4: tcgen05.mma kind::mxf8f6f4 scale_vec::1X
// with E4M3 A and E2M1 B (UE8M0 scales, block 32; K = 32 per instruction).
// and two CTA groupings: cta_group::1 (one SM, 128 x N x 64 per instruction)
// or cta_group::2 (a cluster of two CTAs on two SMs, 256 x N x 64 per
// instruction, issued by the even CTA).
//
// One thread per SM (per pair) issues a long chain of MMAs from shared memory
// (zero operands and scale bytes, or pseudo-random operand bytes with scale
// bytes 120..134) into TMEM and times it with the SM clock.
// Optionally a scale-factor copy (tcgen05.cp) is issued before every group of
// MMAs, as the GEMM main loop does, and optionally the MMAs alternate between
// two accumulators (N <= 128), which separates the accumulator dependency
// from the issue rate.  Optionally the thread also waits, after each group,
// `waits` times on an mbarrier phase that has already completed and commits
// to a second barrier, as a GEMM's MMA thread does once per stage: this
// measures what the issuing thread's own instructions cost the tensor pipe.
//
// Exposed through its own small C entry point in a separate library, used
// only by the benchmark.
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"

namespace fp4lin {
namespace {

constexpr int kMaxN = 256;
constexpr int kSmemUsed = 16384 + kMaxN * 128 + 2048;  // A tile, B tile, scale chunks

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_barrier()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int CTAG>
__device__ __forceinline__ void probe_alloc(uint32_t* slot)
{
    if constexpr (CTAG == 2) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
        tmem_alloc(slot, 512);
        tmem_relinquish();
    }
}

template <int CTAG>
__device__ __forceinline__ void probe_dealloc(uint32_t t)
{
    if constexpr (CTAG == 2)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(t), "r"(512) : "memory");
    else
        tmem_dealloc(t, 512);
}

template <int CTAG>
__device__ __forceinline__ void probe_cp(uint32_t taddr, uint64_t sdesc)
{
    if constexpr (CTAG == 2)
        asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
    else
        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

template <int CTAG>
__device__ __forceinline__ void probe_commit(uint64_t* bar)
{
    if constexpr (CTAG == 2)
        asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         smem_u32(bar))
                     : "memory");
    else
        tc_commit(bar);
}

// One MMA of the given form; `acc` selects accumulate (1) or overwrite (0).
#define FP4_PROBE_MMA(CG, KINDSTR)                                                                          \
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"                                          \
                 "tcgen05.mma.cta_group::" CG ".kind::" KINDSTR " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"( \
                     d),                                                                                    \
                 "l"(ad), "l"(bd), "r"(idesc), "r"(sfa), "r"(sfb), "r"(1u)                                  \
                 : "memory")

template <int KIND, int CTAG>
__device__ __forceinline__ void probe_mma(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t sfa,
                                          uint32_t sfb)
{
    if constexpr (KIND == 4) {
        static_assert(CTAG == 1, "the W4A8 form is probed on one SM");
        FP4_PROBE_MMA("1", "mxf8f6f4.block_scale.scale_vec::1X");
    } else if constexpr (CTAG == 1) {
        if constexpr (KIND == 0)
            FP4_PROBE_MMA("1", "mxf4.block_scale.scale_vec::2X");
        else if constexpr (KIND == 1)
            FP4_PROBE_MMA("1", "mxf4nvf4.block_scale.scale_vec::2X");
        else
            FP4_PROBE_MMA("1", "mxf4nvf4.block_scale.scale_vec::4X");
    } else {
        if constexpr (KIND == 0)
            FP4_PROBE_MMA("2", "mxf4.block_scale.scale_vec::2X");
        else if constexpr (KIND == 1)
            FP4_PROBE_MMA("2", "mxf4nvf4.block_scale.scale_vec::2X");
        else
            FP4_PROBE_MMA("2", "mxf4nvf4.block_scale.scale_vec::4X");
    }
}
#undef FP4_PROBE_MMA

// Instruction descriptor: E2M1 A and B (bits 7-9, 10-12), N >> 3 (17-22),
// scale type (bit 23: 1 = UE8M0, 0 = UE4M3), M >> 4 (24-28).
__host__ __device__ constexpr uint32_t probe_idesc(int kind, uint32_t m, uint32_t n)
{
    if (kind == 4)  // E4M3 A (type 0), E2M1 B (type 5), UE8M0 scales
        return (0u << 7) | (5u << 10) | ((n >> 3) << 17) | (1u << 23) | ((m >> 4) << 24);
    return (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((kind == 3 ? 0u : 1u) << 23) | ((m >> 4) << 24);
}

__device__ __forceinline__ uint32_t probe_hash(uint32_t x)
{
    x ^= x >> 16;
    x *= 0x7feb352du;
    x ^= x >> 15;
    x *= 0x846ca68bu;
    x ^= x >> 16;
    return x;
}

template <int KIND, int CTAG, int N>
__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int iters, int mmas_per_group, int with_cp, int alt,
                                                          int waits, int fill, unsigned long long* cycles,
                                                          unsigned int* status)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* a = smem;                         // 128 rows x 128 B
    uint8_t* b = smem + 16384;                 // N rows x 128 B (cta_group::2: N / 2 rows per CTA)
    uint8_t* sf = smem + 16384 + kMaxN * 128;  // 2 KB of scale chunks
    uint64_t* bar = reinterpret_cast<uint64_t*>(sf + 2048);
    uint64_t* done = bar + 1;  // its phase 0 completes before the chain starts
    uint64_t* sink = bar + 2;  // per-group commits land here; nobody waits on it
    uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 3);
    for (int i = threadIdx.x; i < kSmemUsed / 4; i += blockDim.x) {
        uint32_t v = 0u;
        if (fill) {
            v = probe_hash(static_cast<uint32_t>(i) * 2654435761u + blockIdx.x);
            if (i * 4 >= 16384 + kMaxN * 128) {  // scale bytes: 120 ... 134
                uint32_t w = 0u;
                for (int j = 0; j < 4; ++j)
                    w |= (120u + ((v >> (8 * j)) & 0xFFu) % 15u) << (8 * j);
                v = w;
            }
        }
        reinterpret_cast<uint32_t*>(smem)[i] = v;
    }
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        mbar_init(done, 1);
        mbar_init(sink, 1);
        fence_mbar_init();
        mbar_arrive(done);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const int warp = threadIdx.x >> 5;
    if (warp == 0)
        probe_alloc<CTAG>(slot);
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (CTAG == 2)
        cluster_barrier();  // the peer's shared memory and TMEM are ready before the pair's MMAs read them
    tc_fence_after_sync();
    const uint32_t tmem = *slot;
    const bool issuer = threadIdx.x == 0 && (CTAG == 1 || cluster_rank() == 0);
    if (issuer) {
        constexpr uint32_t M = 128 * CTAG;
        const uint32_t idesc = probe_idesc(KIND, M, N);
        const uint32_t a_s = smem_u32(a), b_s = smem_u32(b), sf_s = smem_u32(sf);
        // accumulators in columns 0-255 (one of N columns, or two of at most
        // 128 alternating); scale columns after them: 16 for A, 32 for B
        const uint32_t sfa_t = tmem + 256;
        const uint32_t sfb_t = sfa_t + 16;
        // the scale columns must hold defined bytes before the first MMA
        for (int g = 0; g < 4; ++g)
            probe_cp<CTAG>(sfa_t + 4 * g, smem_desc(sf_s, 0, 128, 0));
        for (int g = 0; g < 8; ++g)
            probe_cp<CTAG>(sfb_t + 4 * g, smem_desc(sf_s, 0, 128, 0));
        // every operand of the chain is formed before the clock starts, so that the
        // issuing thread does no arithmetic per MMA (it would otherwise pace
        // the narrower MMAs)
        uint64_t ad[4], bd[4];
        uint32_t id[4];
        for (int k = 0; k < 4; ++k) {
            ad[k] = smem_desc(a_s + 32 * k, 16, 1024, 2);
            bd[k] = smem_desc(b_s + 32 * k, 16, 1024, 2);
            // scale selector: two scales per K = 64 step (2X), one per K = 32 step (1X: byte k % 4)
            const uint32_t sel = KIND == 4 ? static_cast<uint32_t>(k) : (KIND >= 2 ? 0u : static_cast<uint32_t>(k & 1) * 2u);
            id[k] = idesc | (sel << 4) | (sel << 29);
        }
        const uint32_t dd[2] = {tmem, tmem + (alt ? 128u : 0u)};
        const uint32_t sa[2] = {sfa_t, sfa_t + 4};
        const uint32_t sb[2] = {sfb_t, sfb_t + 8};
        auto mma = [&](int k) { probe_mma<KIND, CTAG>(dd[k & 1], ad[k & 3], bd[k & 3], id[k & 3], sa[k & 1], sb[k & 1]); };
        auto generic = [&](int k) {
            const uint32_t sel = KIND == 4 ? static_cast<uint32_t>(k & 3)
                                           : (KIND >= 2 ? 0u : static_cast<uint32_t>(k & 1) * 2u);
            probe_mma<KIND, CTAG>(tmem + ((alt && (k & 1)) ? 128u : 0u), smem_desc(a_s + 32 * (k & 3), 16, 1024, 2),
                                  smem_desc(b_s + 32 * (k & 3), 16, 1024, 2), idesc | (sel << 4) | (sel << 29),
                                  sfa_t + 4 * (k & 1), sfb_t + 8 * (k & 1));
        };
        const long long t0 = clock64();
        // one loop per configuration: code for the options a run does not use
        // stays out of the loop (a wait the loop merely contains slows it)
        if (!with_cp && waits == 0 && mmas_per_group == 4) {
            for (int it = 0; it < iters; ++it) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma(k);
            }
        } else if (!with_cp && waits == 0 && mmas_per_group == 8) {
            for (int it = 0; it < iters; ++it) {
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma(k);
            }
        } else if (waits == 0 && mmas_per_group == 4) {
            for (int it = 0; it < iters; ++it) {
                probe_cp<CTAG>(sfa_t + 4 * (it & 1), smem_desc(sf_s + 512, 0, 128, 0));
                probe_cp<CTAG>(sfb_t + 8 * (it & 1), smem_desc(sf_s + 1024, 0, 128, 0));
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma(k);
            }
        } else if (!with_cp && mmas_per_group == 8) {
            for (int it = 0; it < iters; ++it) {
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma(k);
                probe_commit<CTAG>(sink);
                for (int w = 0; w < waits; ++w)
                    mbar_wait_bounded(done, 0, status, 1u, 1000000000ull);
                tc_fence_after_sync();
            }
        } else {
            for (int it = 0; it < iters; ++it) {
                if (with_cp) {
                    probe_cp<CTAG>(sfa_t + 4 * (it & 1), smem_desc(sf_s + 512, 0, 128, 0));
                    probe_cp<CTAG>(sfb_t + 8 * (it & 1), smem_desc(sf_s + 1024, 0, 128, 0));
                }
                for (int k = 0; k < mmas_per_group; ++k)
                    generic(k);
                if (waits > 0) {
                    probe_commit<CTAG>(sink);
                    for (int w = 0; w < waits; ++w)
                        mbar_wait_bounded(done, 0, status, 1u, 1000000000ull);
                    tc_fence_after_sync();
                }
            }
        }
        probe_commit<CTAG>(bar);
        mbar_wait_bounded(bar, 0, status, 1u, 2000000000ull);
        const long long t1 = clock64();
        cycles[blockIdx.x / CTAG] = static_cast<unsigned long long>(t1 - t0);
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (CTAG == 2)
        cluster_barrier();  // the pair's MMAs have finished before either CTA frees its TMEM
    if (warp == 0) {
        tc_fence_after_sync();
        probe_dealloc<CTAG>(tmem);
    }
}

template <int KIND, int CTAG, int N>
cudaError_t run_probe(int iters, int mmas_per_group, int with_cp, int alt, int waits, int fill, int num_ctas,
                      unsigned long long* cycles, unsigned int* status, cudaStream_t s)
{
    const size_t smem = kSmemUsed + 64 + 1024;
    auto kern = mma_peak_kernel<KIND, CTAG, N>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess)
        return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_ctas / CTAG * CTAG);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CTAG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, iters, mmas_per_group, with_cp, alt, waits, fill, cycles, status);
}

}  // namespace
}  // namespace fp4lin

// kind: 0..4 as above; ctag: 1 or 2 (kind 4: 1); n: 128 or 256, and 16, 32
// or 64 for kinds 0 and 4 on one SM (the decode tile widths).  waits: completed
// barrier waits (plus one commit) per group of MMAs; fill: 1 for pseudo-random
// operands.  cycles_dev holds one entry per issuing CTA (num_ctas / ctag).
// Returns a cudaError_t.
extern "C" __attribute__((visibility("default"))) int fp4_mma_peak_probe3(int kind, int ctag, int n, int iters,
                                                                        int mmas_per_group, int with_cp, int alt,
                                                                        int waits, int fill, int num_ctas,
                                                                        unsigned long long* cycles_dev,
                                                                        unsigned int* status_dev, void* stream)
{
    using namespace fp4lin;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (alt && n > 128)
        return static_cast<int>(cudaErrorInvalidValue);  // two accumulators of n columns must leave room for scales
#define FP4_PEAK_CASE(K, G, NN)                                                                     \
    if (kind == K && ctag == G && n == NN)                                                          \
        return static_cast<int>(run_probe<K, G, NN>(iters, mmas_per_group, with_cp, alt, waits, fill, num_ctas, \
                                                    cycles_dev, status_dev, s));
#define FP4_PEAK_KIND(K)     \
    FP4_PEAK_CASE(K, 1, 128) \
    FP4_PEAK_CASE(K, 1, 256) \
    FP4_PEAK_CASE(K, 2, 128) \
    FP4_PEAK_CASE(K, 2, 256)
    FP4_PEAK_KIND(0)
    FP4_PEAK_KIND(1)
    FP4_PEAK_KIND(2)
    FP4_PEAK_KIND(3)
    FP4_PEAK_CASE(0, 1, 16)
    FP4_PEAK_CASE(0, 1, 32)
    FP4_PEAK_CASE(0, 1, 64)
    FP4_PEAK_CASE(4, 1, 16)
    FP4_PEAK_CASE(4, 1, 32)
    FP4_PEAK_CASE(4, 1, 64)
    FP4_PEAK_CASE(4, 1, 128)
    FP4_PEAK_CASE(4, 1, 256)
#undef FP4_PEAK_KIND
#undef FP4_PEAK_CASE
    return static_cast<int>(cudaErrorInvalidValue);
}

// Without the per-group waits, zero operands.
extern "C" __attribute__((visibility("default"))) int fp4_mma_peak_probe2(int kind, int ctag, int n, int iters,
                                                                        int mmas_per_group, int with_cp, int alt,
                                                                        int num_ctas, unsigned long long* cycles_dev,
                                                                        unsigned int* status_dev, void* stream)
{
    return fp4_mma_peak_probe3(kind, ctag, n, iters, mmas_per_group, with_cp, alt, 0, 0, num_ctas, cycles_dev,
                               status_dev, stream);
}

// The original entry point: kind::mxf4, cta_group::1.
extern "C" __attribute__((visibility("default"))) int fp4_mma_peak_probe(int n, int iters, int mmas_per_group,
                                                                       int with_cp, int num_ctas,
                                                                       unsigned long long* cycles_dev,
                                                                       unsigned int* status_dev, void* stream)
{
    return fp4_mma_peak_probe2(0, 1, n, iters, mmas_per_group, with_cp, 0, num_ctas, cycles_dev, status_dev, stream);
}
