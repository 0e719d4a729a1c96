// gemm.cu -- W4A4 block-scaled FP4 GEMM on the 5th-generation tensor cores.
//
//   out[m, n] = bf16_rne( sum_k A[m, k] * B[n, k] + bias[n] )
//
// Both operands are MXFP4 ("Efficiently Serving NVFP4 Models on AMD
// Instinct MI350X/MI355X ... via Online NVFP4 to Quark MXFP4
// Requantization", "Native FP4 matmul": dense layers and MoE experts run on
// native block-scaled FP4 matrix instructions with no separate dequantize
// step); the bf16 output with a bf16 per-output-channel bias follows "W4A4
// MXFP4 Quantization" (Configuration) and "[SGLang] FP4 ..." (section 6).
//
// Design (one CTA per 128 x BN output tile, 6 warps):
//   warp 0      TMA producer: A and B tiles (128-byte swizzled, 128 packed
//               bytes = 256 K-elements per stage) by tensor-map loads, the
//               matching 512-byte scale-factor chunks by bulk copies, all
//               completing on the stage's `full` mbarrier.
//   warp 1      TMEM allocator and MMA issuer: per stage, tcgen05.cp moves the
//               scale chunks into TMEM, then four tcgen05.mma kind::mxf4
//               (K = 64 each, two E8M0 scales per row per instruction)
//               accumulate into a 128 x BN fp32 TMEM tile; tcgen05.commit
//               frees the stage.
//   warps 2-5   epilogue: tcgen05.ld of the accumulator (each warp reads the
//               32 TMEM lanes it may access), + bias, bf16 round, store.
// Every mbarrier wait is bounded; on expiry the kernel records a timeout in
// the status word and winds down without further waits on that path.
#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace fp4lin {

namespace {

constexpr int BM = 128;
constexpr int kStageKBytes = 128;  // packed bytes of K per row per stage (256 elements)
constexpr int kThreads = 192;

struct GemmParams {
    const uint8_t* sfa;
    const uint8_t* sfb;
    const __nv_bfloat16* bias;
    __nv_bfloat16* out;
    const int32_t* offsets;
    int E;
    int M, N, K;
    int kb4;        // K / 128: scale-factor column groups per row tile
    int m_tiles;    // dense: ceil(M/128); grouped: bound on sum_e ceil(rows_e/128)
    int64_t sfb_expert_stride;
    unsigned int* status;
};

template <int BN, int STAGES>
struct Cfg {
    static constexpr int A_BYTES = BM * kStageKBytes;
    static constexpr int B_BYTES = BN * kStageKBytes;
    static constexpr int SFA_BYTES = 1024;             // 128 rows x 2 groups of 4 blocks
    static constexpr int SFB_BYTES = (BN / 128) * 1024;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
    static constexpr int OFF_BAR = OFF_SFB + STAGES * SFB_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 1;
    static constexpr int OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_PREFIX = OFF_TMEM_SLOT + 16;
    static constexpr int SMEM_FIXED = OFF_PREFIX + 1024;  // + 1 KB alignment slack
    // TMEM columns: accumulator, then two scale-factor buffers (stage parity)
    static constexpr int SF_COLS_A = 8;                    // 2 groups x 4 columns
    static constexpr int SF_COLS_B_GROUP = 4 * (BN / 128);
    static constexpr int SF_COLS = SF_COLS_A + 2 * SF_COLS_B_GROUP;
    static constexpr int TMEM_USED = BN + 2 * SF_COLS;
    static constexpr int TMEM_COLS = TMEM_USED <= 32 ? 32 : TMEM_USED <= 64 ? 64 : TMEM_USED <= 128 ? 128
                                     : TMEM_USED <= 256 ? 256 : 512;
    static_assert(TMEM_USED <= 512, "TMEM overflow");
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

template <int BN, int STAGES, bool kGrouped>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_mxfp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const GemmParams p)
{
    using C = Cfg<BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* empty = full + STAGES;
    uint64_t* accum_full = empty + STAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM_SLOT);
    int32_t* tiles_before = reinterpret_cast<int32_t*>(smem + C::OFF_PREFIX);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ------------------------------------------------------ tile decode
    int n_tile = static_cast<int>(blockIdx.x) / p.m_tiles;
    int g_tile = static_cast<int>(blockIdx.x) % p.m_tiles;
    int expert = 0;
    int64_t a_row0 = static_cast<int64_t>(g_tile) * BM;
    int rows_valid = p.M - static_cast<int>(a_row0);
    if constexpr (kGrouped) {
        if (warp == 0) {
            // exclusive prefix of per-expert 128-row tile counts
            int carry = 0;
            for (int base = 0; base <= p.E; base += 32) {
                const int e = base + lane;
                int t = 0;
                if (e < p.E)
                    t = (__ldg(p.offsets + e + 1) - __ldg(p.offsets + e) + 127) >> 7;
                int incl = t;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                    if (lane >= d)
                        incl += v;
                }
                if (e <= p.E)
                    tiles_before[e] = carry + incl - t;
                carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
            }
        }
        __syncthreads();
        if (g_tile >= tiles_before[p.E])
            return;  // whole CTA: this grid slot has no tile
        int lo = 0, hi = p.E;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (tiles_before[mid] <= g_tile)
                lo = mid;
            else
                hi = mid;
        }
        expert = lo;
        const int start = __ldg(p.offsets + lo);
        const int end = __ldg(p.offsets + lo + 1);
        a_row0 = start + static_cast<int64_t>(g_tile - tiles_before[lo]) * BM;
        rows_valid = end - static_cast<int>(a_row0);
    }
    if (rows_valid > BM)
        rows_valid = BM;
    const int n0 = n_tile * BN;
    const int64_t b_row0 = static_cast<int64_t>(expert) * p.N + n0;
    const uint8_t* sfb = p.sfb + static_cast<int64_t>(expert) * p.sfb_expert_stride;
    const int n_row_tiles_b = (p.N + 127) / 128;
    int nsfb = n_row_tiles_b - n0 / 128;
    if (nsfb > BN / 128)
        nsfb = BN / 128;
    const int nkb = (p.K + 255) / 256;

    // ------------------------------------------------------------ setup
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accum_full, 1);
        fence_mbar_init();
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------- TMA producer
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % STAGES;
            const uint32_t ph = static_cast<uint32_t>(kb / STAGES) & 1u;
            if (!mbar_wait_bounded(&empty[s], ph ^ 1u, p.status, kStatusTimeout, kWaitLimitNs))
                break;
            const int groups = min(2, p.kb4 - 2 * kb);
            const uint32_t sf_bytes = static_cast<uint32_t>(groups) * 512u;
            mbar_arrive_expect_tx(&full[s], C::A_BYTES + C::B_BYTES + sf_bytes * (1u + nsfb));
            tma_load_2d(smem + C::OFF_A + s * C::A_BYTES, &tmA, &full[s], kb * kStageKBytes,
                        static_cast<int32_t>(a_row0));
            tma_load_2d(smem + C::OFF_B + s * C::B_BYTES, &tmB, &full[s], kb * kStageKBytes,
                        static_cast<int32_t>(b_row0));
            bulk_load(smem + C::OFF_SFA + s * C::SFA_BYTES,
                      p.sfa + (static_cast<int64_t>(g_tile) * p.kb4 + 2 * kb) * 512, sf_bytes, &full[s]);
            for (int j = 0; j < nsfb; ++j)
                bulk_load(smem + C::OFF_SFB + s * C::SFB_BYTES + j * 1024,
                          sfb + (static_cast<int64_t>(n0 / 128 + j) * p.kb4 + 2 * kb) * 512, sf_bytes, &full[s]);
        }
    } else if (warp == 1 && lane == 0) {
        // --------------------------------------------------- MMA issuer
        constexpr uint32_t idesc = idesc_mxf4(BM, BN);
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % STAGES;
            const uint32_t ph = static_cast<uint32_t>(kb / STAGES) & 1u;
            if (!mbar_wait_bounded(&full[s], ph, p.status, kStatusTimeout, kWaitLimitNs))
                break;
            tc_fence_after_sync();
            const int groups = min(2, p.kb4 - 2 * kb);
            const uint32_t sfa_t = tmem_base + BN + (kb & 1) * C::SF_COLS;
            const uint32_t sfb_t = sfa_t + C::SF_COLS_A;
            const uint32_t sfa_s = smem_u32(smem + C::OFF_SFA + s * C::SFA_BYTES);
            const uint32_t sfb_s = smem_u32(smem + C::OFF_SFB + s * C::SFB_BYTES);
            for (int g = 0; g < groups; ++g) {
                tc_cp_32x128b_warpx4(sfa_t + 4 * g, smem_desc(sfa_s + 512 * g, 0, 128, 0));
#pragma unroll
                for (int j = 0; j < BN / 128; ++j)
                    tc_cp_32x128b_warpx4(sfb_t + g * C::SF_COLS_B_GROUP + 4 * j,
                                         smem_desc(sfb_s + 1024 * j + 512 * g, 0, 128, 0));
            }
            const uint32_t a_s = smem_u32(smem + C::OFF_A + s * C::A_BYTES);
            const uint32_t b_s = smem_u32(smem + C::OFF_B + s * C::B_BYTES);
            for (int k = 0; k < 2 * groups; ++k) {
                const int g = k >> 1;
                const uint32_t sf_id = static_cast<uint32_t>(k & 1) * 2u;
                tc_mma_mxf4(tmem_base, smem_desc(a_s + 32 * k, 16, 1024, 2), smem_desc(b_s + 32 * k, 16, 1024, 2),
                            idesc_with_sf_id(idesc, sf_id), sfa_t + 4 * g, sfb_t + g * C::SF_COLS_B_GROUP,
                            (kb | k) != 0 ? 1u : 0u);
            }
            tc_commit(&empty[s]);
        }
        tc_commit(accum_full);
    } else if (warp >= 2) {
        // ------------------------------------------------------ epilogue
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const bool ok = mbar_wait_bounded(accum_full, 0u, p.status, kStatusTimeout, kWaitLimitNs);
        tc_fence_after_sync();
        const __nv_bfloat16* bias = p.bias ? p.bias + static_cast<int64_t>(expert) * p.N : nullptr;
        __nv_bfloat16* orow = p.out + (a_row0 + r) * static_cast<int64_t>(p.N);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + 32 * c, v);
            tmem_ld_wait();
            const int col0 = n0 + 32 * c;
            if (!ok || r >= rows_valid || col0 >= p.N)
                continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int col = col0 + 8 * j;
                if (col >= p.N)
                    break;
                float f[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    f[i] = __uint_as_float(v[8 * j + i]);
                if (bias) {
                    const uint4 bb = *reinterpret_cast<const uint4*>(bias + col);
                    const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        f[2 * i] += __uint_as_float(bw[i] << 16);
                        f[2 * i + 1] += __uint_as_float(bw[i] & 0xFFFF0000u);
                    }
                }
                uint4 o;
                o.x = pack_bf16x2(f[0], f[1]);
                o.y = pack_bf16x2(f[2], f[3]);
                o.z = pack_bf16x2(f[4], f[5]);
                o.w = pack_bf16x2(f[6], f[7]);
                *reinterpret_cast<uint4*>(orow + col) = o;
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// --------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// [rows, K/2] packed bytes, box = 128 bytes x box_rows, 128-byte swizzle.
bool make_operand_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kStageKBytes), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int STAGES, bool kGrouped>
cudaError_t launch_tile_kernel(const GemmArgs& a, cudaStream_t stream)
{
    using C = Cfg<BN, STAGES>;
    CUtensorMap tmA, tmB;
    if (!make_operand_map(&tmA, a.a, a.M, a.K, BM))
        return cudaErrorInvalidValue;
    if (!make_operand_map(&tmB, a.b, static_cast<int64_t>(a.E) * a.N, a.K, BN))
        return cudaErrorInvalidValue;
    GemmParams p;
    p.sfa = a.sa;
    p.sfb = a.sb;
    p.bias = static_cast<const __nv_bfloat16*>(a.bias);
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.offsets = a.row_offsets;
    p.E = a.E;
    p.M = static_cast<int>(a.M);
    p.N = static_cast<int>(a.N);
    p.K = static_cast<int>(a.K);
    p.kb4 = static_cast<int>(a.K / 128);
    p.m_tiles = kGrouped ? static_cast<int>((a.M + static_cast<int64_t>(a.E) * 127) / 128)
                         : static_cast<int>((a.M + 127) / 128);
    p.sfb_expert_stride = ((a.N + 127) / 128) * 128 * (a.K / 32);
    p.status = a.status;
    const int n_tiles = static_cast<int>((a.N + BN - 1) / BN);
    const int64_t grid = static_cast<int64_t>(p.m_tiles) * n_tiles;
    if (grid == 0)
        return cudaSuccess;
    const size_t smem = C::SMEM_FIXED + (kGrouped ? sizeof(int32_t) * (a.E + 1) : 0);
    auto kern = gemm_mxfp4_kernel<BN, STAGES, kGrouped>;
    // The shared-memory opt-in is a per-device function attribute: set it
    // once per device (and grow it if a larger grouped prefix needs more).
    static std::mutex mu;
    static size_t configured[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess || dev < 0 || dev >= 64)
        return err != cudaSuccess ? err : cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (configured[dev] < smem) {
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
            if (err != cudaSuccess)
                return err;
            configured[dev] = smem;
        }
    }
    kern<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(tmA, tmB, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t stream)
{
    const bool grouped = a.row_offsets != nullptr;
    // Wide tiles when there are enough of them to fill the machine.
    const int64_t m_tiles = grouped ? (a.M + static_cast<int64_t>(a.E) * 127) / 128 : (a.M + 127) / 128;
    const bool wide = a.N >= 256 && m_tiles * ((a.N + 255) / 256) >= 148;
    if (grouped)
        return wide ? launch_tile_kernel<256, 4, true>(a, stream) : launch_tile_kernel<128, 6, true>(a, stream);
    return wide ? launch_tile_kernel<256, 4, false>(a, stream) : launch_tile_kernel<128, 6, false>(a, stream);
}

}  // namespace fp4lin
