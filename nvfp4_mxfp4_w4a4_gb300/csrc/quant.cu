// quant.cu -- the memory-bound quantizers:
//   * NVFP4 -> MXFP4 requantization (load time, once per layer),
//   * dynamic MXFP4 quantization of bf16 activations (dense and grouped),
//   * the bf16 -> NVFP4 producer.
//
// Method: "Efficiently Serving NVFP4 Models on AMD Instinct MI350X/MI355X
// Accelerators via Online NVFP4 to Quark MXFP4 Requantization" (the online
// requantization pipeline and the serve-time activation path) with the MX
// block rule of "W4A4 MXFP4 Quantization" (Single-Scale Block Scaling
// (OCP / UOS)) and the NVFP4 layout of "[SGLang] FP4 ..." (sections 3-4).
//
// All three kernels stream: each warp owns a (row, chunk) work item, loads
// its whole chunk with 128-bit loads before doing any arithmetic (several
// loads in flight per thread), and writes packed codes with 128/32-bit
// stores.  Scale bytes for the swizzled layout are gathered with shuffles so
// that one lane writes the four bytes of a 4-block group as one 32-bit store.
#include "formats.cuh"
#include "internal.h"

namespace fp4lin {

namespace {

constexpr int kThreads = 256;  // 8 warps per CTA

__device__ __forceinline__ uint4 ld_stream_u4(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_stream_u16(const void* p)
{
    unsigned short v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// ------------------------------------------------------------ requant
// One NVFP4 half-block (16 codes in two 32-bit words, one E4M3 scale)
// contributes its largest magnitude to the block amax.  The largest
// magnitude code is found with a byte-permute one-hot lookup: each 3-bit
// magnitude selects byte m of the constant 0x80..01, the OR of all results
// is the set of magnitudes present.
__device__ __forceinline__ uint32_t max_magnitude_code(uint32_t w0, uint32_t w1)
{
    constexpr uint32_t kOneHotLo = 0x08040201u, kOneHotHi = 0x80402010u;
    const uint32_t m0 = w0 & 0x77777777u, m1 = w1 & 0x77777777u;
    uint32_t p = __byte_perm(kOneHotLo, kOneHotHi, m0) | __byte_perm(kOneHotLo, kOneHotHi, m0 >> 16) |
                 __byte_perm(kOneHotLo, kOneHotHi, m1) | __byte_perm(kOneHotLo, kOneHotHi, m1 >> 16);
    p |= p >> 16;
    p |= p >> 8;
    return 31u - __clz(p & 0xFFu);
}

// Output codes of one half-block as an 8-entry map magnitude -> code.  With
// S = |E4M3 scale| and ag = |g|, the decoded magnitude of code m is
// RN(G[m] * S * ag).  The products with G in {0.5, 1, 1.5} are each rounded
// once (H, P, Q); G in {2, 4} and {3, 6} are exact doublings of P and Q
// (their overflow matches that of the direct product).  Multiplying by 2^-e
// is exact except in deep underflow, where every code is 0 anyway.  The map
// is returned as bytes 0..7 of (t0, t1) for byte-permute lookups.
__device__ __forceinline__ void half_block_code_map(float S, float ag, float se, uint32_t& t0, uint32_t& t1)
{
    const float H = __fmul_rn(0.5f * S, ag);
    const float P = __fmul_rn(S, ag);
    const float Q = __fmul_rn(1.5f * S, ag);
    const float h = __fmul_rn(H, se), x = __fmul_rn(P, se), y = __fmul_rn(Q, se);
    const uint32_t r1 = __float_as_uint(e2m1_code_scaled<0>(h));
    const uint32_t r2 = __float_as_uint(e2m1_code_scaled<0>(x));
    const uint32_t r3 = __float_as_uint(e2m1_code_scaled<0>(y));
    const uint32_t r4 = __float_as_uint(e2m1_code_scaled<1>(x));
    const uint32_t r5 = __float_as_uint(e2m1_code_scaled<1>(y));
    const uint32_t r6 = __float_as_uint(e2m1_code_scaled<2>(x));
    const uint32_t r7 = __float_as_uint(e2m1_code_scaled<2>(y));
    // byte 1 of kMagic + code is 0x00: use it for the code of magnitude 0
    const uint32_t a = __byte_perm(r1, r2, 0x1401u);  // [0, r1, r2, -]
    t0 = __byte_perm(a, r3, 0x4210u);                  // [0, r1, r2, r3]
    const uint32_t b = __byte_perm(r4, r5, 0x0040u);  // [r4, r5, -, -]
    const uint32_t c = __byte_perm(r6, r7, 0x4000u);  // [-, -, r6, r7]
    t1 = __byte_perm(b, c, 0x7610u);                   // [r4, r5, r6, r7]
}

// Apply the magnitude map to 8 codes in one word and restore the signs
// (flipped when the scale times g is negative).
__device__ __forceinline__ uint32_t apply_code_map(uint32_t w, uint32_t t0, uint32_t t1, uint32_t flip)
{
    const uint32_t m = w & 0x77777777u;
    const uint32_t lo = __byte_perm(t0, t1, m);
    const uint32_t hi = __byte_perm(t0, t1, m >> 16);
    const uint32_t a = lo | (lo >> 4);
    const uint32_t b = hi | (hi >> 4);
    return __byte_perm(a, b, 0x6420u) | ((w & 0x88888888u) ^ flip);
}

// One 32-element NVFP4 block (16 code bytes, two E4M3 scales) -> MXFP4.
__device__ __forceinline__ void requant_block(uint4 codes, uint32_t scales, float ag, uint32_t gsign, int uos,
                                              uint4& out, uint32_t& sf)
{
    const float2 s = e4m3x2_to_float2(scales);
    const float S0 = fabsf(s.x), S1 = fabsf(s.y);
    const uint32_t mm0 = max_magnitude_code(codes.x, codes.y);
    const uint32_t mm1 = max_magnitude_code(codes.z, codes.w);
    const float amax0 = __fmul_rn(__fmul_rn(e2m1_mag_value(mm0), S0), ag);
    const float amax1 = __fmul_rn(__fmul_rn(e2m1_mag_value(mm1), S1), ag);
    const uint32_t ab = max(__float_as_uint(amax0), __float_as_uint(amax1));
    if (ab >= 0x7F800000u) {  // NaN or Inf somewhere in the block
        out = make_uint4(0u, 0u, 0u, 0u);
        sf = 0xFFu;
        return;
    }
    const int e = mx_shared_exp(ab, uos);
    sf = static_cast<uint32_t>(e + 127);
    const float se = exp2_neg(e);
    const uint32_t f0 = ((__float_as_uint(s.x) >> 31) ^ gsign) ? 0x88888888u : 0u;
    const uint32_t f1 = ((__float_as_uint(s.y) >> 31) ^ gsign) ? 0x88888888u : 0u;
    uint32_t t0, t1;
    half_block_code_map(S0, ag, se, t0, t1);
    out.x = apply_code_map(codes.x, t0, t1, f0);
    out.y = apply_code_map(codes.y, t0, t1, f0);
    half_block_code_map(S1, ag, se, t0, t1);
    out.z = apply_code_map(codes.z, t0, t1, f1);
    out.w = apply_code_map(codes.w, t0, t1, f1);
}

// Work item = (row, chunk of 32*U consecutive blocks); lane owns block
// c = chunk*32*U + 32*u + lane.  Rows run over the padded row count when the
// scales are swizzled so that pad rows and pad block columns get zero bytes.
template <int U>
__global__ void __launch_bounds__(kThreads) requant_kernel(const uint8_t* __restrict__ wp,
                                                           const uint8_t* __restrict__ ws, float g,
                                                           uint8_t* __restrict__ op, uint8_t* __restrict__ osf,
                                                           int64_t N, int64_t K, int64_t rows, int kb, int kbp,
                                                           int nch, int uos, int swizzled)
{
    const int lane = threadIdx.x & 31;
    const int64_t item = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t row = item / nch;
    if (row >= rows)
        return;
    const int c0 = static_cast<int>(item - row * nch) * 32 * U + lane;
    const bool row_real = row < N;
    const float ag = fabsf(g);
    const uint32_t gsign = __float_as_uint(g) >> 31;
    const uint8_t* wrow = wp + row * (K / 2);
    const uint8_t* srow = ws + row * (K / 16);

    uint4 codes[U];
    uint32_t sc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u;
        if (row_real && c < kb) {
            codes[u] = ld_stream_u4(wrow + static_cast<int64_t>(c) * 16);
            sc[u] = ld_stream_u16(srow + static_cast<int64_t>(c) * 2);
        } else {
            codes[u] = make_uint4(0u, 0u, 0u, 0u);
            sc[u] = 0u;
        }
    }
    const int64_t kb4 = kbp >> 2;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u;
        const bool real = row_real && c < kb;
        uint4 out;
        uint32_t sf;
        requant_block(codes[u], sc[u], ag, gsign, uos, out, sf);
        if (real)
            *reinterpret_cast<uint4*>(op + row * (K / 2) + static_cast<int64_t>(c) * 16) = out;
        if (!real)
            sf = 0u;
        if (swizzled) {
            const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, sf, 1);
            const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, sf, 2);
            const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, sf, 3);
            if ((lane & 3) == 0 && c < kbp)
                *reinterpret_cast<uint32_t*>(osf + sf_swizzled_offset(row, c, kb4)) =
                    sf | (b1 << 8) | (b2 << 16) | (b3 << 24);
        } else if (real) {
            osf[row * kb + c] = static_cast<uint8_t>(sf);
        }
    }
}

// ------------------------------------------------------- activation quant
// One lane holds 8 consecutive bf16 of a 32-element block (4 lanes per
// block).  Returns the packed codes (4 bytes) and, through `sf`, the block's
// scale byte (the same on all 4 lanes).
__device__ __forceinline__ uint32_t act_quant_lane(uint4 v, int uos, uint32_t& sf)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    // amax as bf16 bit patterns of |x| (NaN above Inf above every finite)
    const uint32_t a = __vmaxu2(__vmaxu2(w[0] & 0x7FFF7FFFu, w[1] & 0x7FFF7FFFu),
                                __vmaxu2(w[2] & 0x7FFF7FFFu, w[3] & 0x7FFF7FFFu));
    uint32_t am = max(a & 0xFFFFu, a >> 16);
    am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
    am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
    const uint32_t ab = am << 16;
    if (ab >= 0x7F800000u) {
        sf = 0xFFu;
        return 0u;
    }
    const int e = mx_shared_exp(ab, uos);
    sf = static_cast<uint32_t>(e + 127);
    const float se = exp2_neg(e);
    uint32_t packed = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float xl = __uint_as_float(w[j] << 16);
        const float xh = __uint_as_float(w[j] & 0xFFFF0000u);
        const uint32_t cl = e2m1_code(__fmul_rn(fabsf(xl), se)) | ((w[j] >> 12) & 0x8u);
        const uint32_t ch = e2m1_code(__fmul_rn(fabsf(xh), se)) | ((w[j] >> 28) & 0x8u);
        packed |= (cl | (ch << 4)) << (8 * j);
    }
    return packed;
}

// Tile-prefix of a grouped activation tensor: group e starts at scale row
// 128 * tiles_before[e].  Computed by one warp into shared memory.
__device__ void group_tile_prefix(const int32_t* offsets, int E, int32_t* tiles_before)
{
    const int lane = threadIdx.x & 31;
    int carry = 0;
    for (int base = 0; base <= E; base += 32) {
        const int e = base + lane;
        int t = 0;
        if (e < E)
            t = (__ldg(offsets + e + 1) - __ldg(offsets + e) + 127) >> 7;
        int incl = t;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int n = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= d)
                incl += n;
        }
        if (e <= E)
            tiles_before[e] = carry + incl - t;
        carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
}

// Work item = (scale row, chunk of 8*U blocks).  For the dense tensor the
// scale row is the activation row (rows >= M are pad rows).  For the grouped
// tensor scale rows live in the padded per-group space; `grouped` selects
// the mapping.  Lane owns quarter (lane & 3) of block chunk*8U + 8u + lane/4.
template <int U, bool kGrouped>
__global__ void __launch_bounds__(kThreads) act_quant_kernel(const uint16_t* __restrict__ x,
                                                             uint8_t* __restrict__ op, uint8_t* __restrict__ osf,
                                                             int64_t M, int64_t K, int64_t sf_rows, int kb,
                                                             int kbp, int nch, int uos, int swizzled,
                                                             const int32_t* __restrict__ offsets, int E)
{
    extern __shared__ int32_t tiles_before[];
    if (kGrouped) {
        if (threadIdx.x < 32)
            group_tile_prefix(offsets, E, tiles_before);
        __syncthreads();
    }
    const int lane = threadIdx.x & 31;
    const int64_t item = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t srow = item / nch;
    if (srow >= sf_rows)
        return;
    int64_t xrow = srow;
    bool row_real = srow < M;
    if (kGrouped) {
        // locate the group whose padded tile range holds this scale row
        const int tile = static_cast<int>(srow >> 7);
        if (tile >= tiles_before[E])
            return;
        int lo = 0, hi = E;  // invariant: tiles_before[lo] <= tile < tiles_before[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (tiles_before[mid] <= tile)
                lo = mid;
            else
                hi = mid;
        }
        const int64_t local = srow - static_cast<int64_t>(tiles_before[lo]) * 128;
        const int64_t start = __ldg(offsets + lo), rows_e = __ldg(offsets + lo + 1) - start;
        row_real = local < rows_e;
        xrow = start + local;
    }
    const int q = lane & 3;
    const int cbase = static_cast<int>(item - srow * nch) * 8 * U + (lane >> 2);
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int c = cbase + 8 * u;
        if (row_real && c < kb)
            v[u] = ld_stream_u4(x + xrow * K + static_cast<int64_t>(c) * 32 + q * 8);
        else
            v[u] = make_uint4(0u, 0u, 0u, 0u);
    }
    const int64_t kb4 = kbp >> 2;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int c = cbase + 8 * u;
        const bool real = row_real && c < kb;
        uint32_t sf;
        const uint32_t packed = act_quant_lane(v[u], uos, sf);
        if (real)
            *reinterpret_cast<uint32_t*>(op + xrow * (K / 2) + static_cast<int64_t>(c) * 16 + q * 4) = packed;
        if (!real)
            sf = 0u;
        if (swizzled) {
            const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, sf, 4);
            const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, sf, 8);
            const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, sf, 12);
            if ((lane & 15) == 0 && c < kbp)
                *reinterpret_cast<uint32_t*>(osf + sf_swizzled_offset(srow, c, kb4)) =
                    sf | (b1 << 8) | (b2 << 16) | (b3 << 24);
        } else if (real && q == 0) {
            osf[xrow * kb + c] = static_cast<uint8_t>(sf);
        }
    }
}

// ------------------------------------------------------- NVFP4 producer
// One thread per 8 consecutive bf16 (two threads per 16-element block).
__global__ void __launch_bounds__(kThreads) quant_nvfp4_kernel(const uint16_t* __restrict__ x, float g,
                                                               uint8_t* __restrict__ op,
                                                               uint8_t* __restrict__ osf, int64_t groups,
                                                               int64_t K)
{
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    // both threads of a block stay active for the shuffle; t / 2 indexes blocks
    const bool active = t < groups;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    const int64_t tt = active ? t : 0;
    if (active)
        v = ld_stream_u4(x + tt * 8);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const uint32_t a = __vmaxu2(__vmaxu2(w[0] & 0x7FFF7FFFu, w[1] & 0x7FFF7FFFu),
                                __vmaxu2(w[2] & 0x7FFF7FFFu, w[3] & 0x7FFF7FFFu));
    uint32_t am = max(a & 0xFFFFu, a >> 16);
    am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
    const float bamax = __uint_as_float(am << 16);
    const float d6 = __fmul_rn(6.0f, g);
    const float tq = __fdiv_rn(bamax, d6);
    const uint32_t sb = float_to_e4m3_satfinite(tq);
    const float den = __fmul_rn(e4m3x2_to_float2(sb).x, g);
    const bool zero_codes = (den == 0.0f) || (den != den);
    uint32_t packed = 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t bits = (j & 1) ? (w[j >> 1] & 0xFFFF0000u) : (w[j >> 1] << 16);
        const float xv = __uint_as_float(bits);
        uint32_t code;
        if (zero_codes) {
            code = (bits >> 28) & 0x8u;
        } else {
            const float qv = __fdiv_rn(xv, den);
            code = e2m1_code(fabsf(qv)) | ((__float_as_uint(qv) >> 28) & 0x8u);
        }
        packed |= code << (4 * j);
    }
    if (active) {
        *reinterpret_cast<uint32_t*>(op + tt * 4) = packed;
        if ((tt & 1) == 0)
            osf[tt >> 1] = static_cast<uint8_t>(sb);
    }
    (void)K;
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

// ------------------------------------------------------------- launchers
cudaError_t launch_requant(const uint8_t* wp, const uint8_t* ws, float g, uint8_t* op, uint8_t* osf, int64_t N,
                           int64_t K, int alg, int swizzled, cudaStream_t stream)
{
    constexpr int U = 4;
    const int kb = static_cast<int>(K / 32);
    const int kbp = swizzled ? static_cast<int>(ceil_div(kb, 4) * 4) : kb;
    const int64_t rows = swizzled ? ceil_div(N, 128) * 128 : N;
    const int nch = static_cast<int>(ceil_div(kbp, 32 * U));
    const int64_t warps = rows * nch;
    const int64_t blocks = ceil_div(warps * 32, kThreads);
    requant_kernel<U><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
        wp, ws, g, op, osf, N, K, rows, kb, kbp, nch, alg == 2 ? 1 : 0, swizzled);
    return cudaGetLastError();
}

cudaError_t launch_act_quant(const void* x, uint8_t* op, uint8_t* osf, int64_t M, int64_t K, int alg,
                             int swizzled, cudaStream_t stream)
{
    constexpr int U = 4;
    const int kb = static_cast<int>(K / 32);
    const int kbp = swizzled ? static_cast<int>(ceil_div(kb, 4) * 4) : kb;
    const int64_t rows = swizzled ? ceil_div(M, 128) * 128 : M;
    const int nch = static_cast<int>(ceil_div(kbp, 8 * U));
    const int64_t blocks = ceil_div(rows * nch * 32, kThreads);
    if (blocks == 0)
        return cudaSuccess;
    act_quant_kernel<U, false><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
        static_cast<const uint16_t*>(x), op, osf, M, K, rows, kb, kbp, nch, alg == 2 ? 1 : 0, swizzled, nullptr,
        0);
    return cudaGetLastError();
}

cudaError_t launch_act_quant_grouped(const void* x, const int32_t* offsets, int E, int64_t total_M, int64_t K,
                                     uint8_t* op, uint8_t* osf, int alg, cudaStream_t stream)
{
    constexpr int U = 4;
    const int kb = static_cast<int>(K / 32);
    const int kbp = static_cast<int>(ceil_div(kb, 4) * 4);
    const int64_t rows = ((total_M + static_cast<int64_t>(E) * 127) / 128) * 128;  // bound on padded rows
    const int nch = static_cast<int>(ceil_div(kbp, 8 * U));
    const int64_t blocks = ceil_div(rows * nch * 32, kThreads);
    if (blocks == 0)
        return cudaSuccess;
    const size_t smem = sizeof(int32_t) * static_cast<size_t>(E + 1);
    act_quant_kernel<U, true><<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(
        static_cast<const uint16_t*>(x), op, osf, total_M, K, rows, kb, kbp, nch, alg == 2 ? 1 : 0, 1, offsets,
        E);
    return cudaGetLastError();
}

cudaError_t launch_quant_nvfp4(const void* x, float g, uint8_t* op, uint8_t* osf, int64_t M, int64_t K,
                               cudaStream_t stream)
{
    const int64_t groups = M * K / 8;
    const int64_t blocks = ceil_div(groups, kThreads);
    if (blocks == 0)
        return cudaSuccess;
    quant_nvfp4_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(static_cast<const uint16_t*>(x), g,
                                                                                op, osf, groups, K);
    return cudaGetLastError();
}

}  // namespace fp4lin
