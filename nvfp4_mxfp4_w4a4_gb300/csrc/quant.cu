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
#include <algorithm>
#include <mutex>

#include "formats.cuh"
#include "ptx.cuh"
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
//
// Work split: a lane owns 4 consecutive 32-element blocks of a row (64 code
// bytes, 8 E4M3 bytes); a warp owns a chunk of 128 blocks of one row; the
// grid is persistent and walks (row, chunk) items with the next item's loads
// in flight while the current one is converted.  The 4 scale bytes a lane
// produces are one 32-bit word of the swizzled layout.
//
// Per half-block (16 codes, one scale s) the output codes come from an
// 8-entry map magnitude -> code, applied to 8 nibbles at once with byte
// permutes.  The maps depend only on (s, e - er(s)) for a tensor (fixed g)
// and are tabulated per CTA in shared memory at kernel start.

__device__ __forceinline__ void ld_nc_v8(const void* p, uint32_t (&r)[8])
{
    asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "l"(p));
}

__device__ __forceinline__ void st_v8(void* p, const uint32_t (&r)[8])
{
    asm volatile("st.global.v8.u32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(r[0]), "r"(r[1]),
                 "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ uint2 ld_nc_u64(const void* p)
{
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_nc_u4_cached(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Packs the codes of magnitudes 1..7 (each the low byte of kMagic + code)
// into the two permute-table words [0, r1, r2, r3], [r4, r5, r6, r7].  Byte 1
// of kMagic + code is 0x00 and supplies the code of magnitude 0.
__device__ __forceinline__ uint2 pack_code_map(uint32_t r1, uint32_t r2, uint32_t r3, uint32_t r4, uint32_t r5,
                                               uint32_t r6, uint32_t r7)
{
    const uint32_t a = __byte_perm(r1, r2, 0x1401u);
    const uint32_t b = __byte_perm(r4, r5, 0x0040u);
    const uint32_t c = __byte_perm(r6, r7, 0x4000u);
    return make_uint2(__byte_perm(a, r3, 0x4210u), __byte_perm(b, c, 0x7610u));
}

// Code maps for one tensor (fixed global scale g).  Entry (s, d) holds the
// map of a half-block with E4M3 scale byte s (sign cleared) when the block
// exponent is e = er(s) + d, er(s) the unbiased exponent of P, d in [-3, 5].
// With S = value(s), the decoded magnitude of code k is D(k) =
// RN(E2M1(k) S |g|), rounded once more to bf16 when the intermediate is bf16:
// H, P, Q for codes 1..3.  For codes 4..7, D is 2P, 2Q, 4P, 4Q exactly when
// S |g| >= 2^-125 (doubling commutes with rounding to a normal float32 or
// bf16 value, overflow included); below that the products are subnormal,
// where a doubled rounded value can sit one ulp from the rounded double, so
// those four are rounded one by one.  Multiplying by 2^-e is exact except in
// deep underflow, where every code is 0 anyway.  A half whose largest code
// is m >= 1 has amax >= H, so its block exponent is >= er - 3; at d >= 6
// every magnitude is below 2^(e-2) and maps to 0 (entry 9).  A half of zero
// codes reads 0 from any entry.  Exponents outside [-127, 126] never occur
// for a finite block and stay 0.  Each entry is built by its own thread:
// three products scaled by 2^-e and seven code roundings (the doublings for
// codes 4..7 happen inside the rounding's fused multiply-adds).
constexpr int kMapD = 10;
constexpr int kMapEntries = 128 * kMapD;

// Per-tensor tables beside the code maps (all for the tensor's |g|):
//   texp[s * 8 + m]  biased block exponent (e + 127) that a half with scale
//                    byte s and largest magnitude code m asks for, from its
//                    amax RN(E2M1(m) S |g|) by the scale rule; 255 when that
//                    amax is NaN or Inf.  The rule is monotone in amax, so a
//                    block's exponent is the larger of its halves' entries.
//   ter[s]           biased exponent of RN(S |g|), which places the block
//                    exponent among the scale's code maps.
struct RequantTables {
    uint2 map[kMapEntries];
    uint8_t texp[128 * 8];
    uint8_t ter[128];
};

// Table options: the block rule and the precision of the decoded values.
constexpr int kRuleUos = 1;   // UOS block rule (else OCP)
constexpr int kRuleBf16 = 2;  // decoded values rounded to bf16 before the block rule

__device__ __forceinline__ float round_to_bf16(float x)
{
    return __bfloat162float(__float2bfloat16_rn(x));
}

__device__ void build_code_maps(float ag, int rule, RequantTables& tb)
{
    const int uos = rule & kRuleUos;
    const bool bf16 = (rule & kRuleBf16) != 0;
    // decoded magnitude from an exact E2M1 x E4M3 product: one float32
    // rounding, then bf16 for the bf16 intermediate
    auto decode = [&](float cs) {
        const float v = __fmul_rn(cs, ag);
        return bf16 ? round_to_bf16(v) : v;
    };
    for (int i = threadIdx.x; i < 128 * 8; i += blockDim.x) {
        const float S = fabsf(e4m3x2_to_float2(static_cast<uint32_t>(i >> 3)).x);
        const float amax = decode(__fmul_rn(e2m1_mag_value(static_cast<uint32_t>(i & 7)), S));
        const uint32_t ab = __float_as_uint(amax);
        tb.texp[i] = ab >= 0x7F800000u ? uint8_t(255) : static_cast<uint8_t>(mx_shared_exp(ab, uos) + 127);
    }
    // one thread per entry (scale byte sb, d = di - 3)
    for (int i = threadIdx.x; i < kMapEntries; i += blockDim.x) {
        const int sb = i / kMapD, di = i - sb * kMapD;
        const float S = e4m3x2_to_float2(static_cast<uint32_t>(sb)).x;
        const float P = decode(S);
        const int er = static_cast<int>(__float_as_uint(P) >> 23) - 127;
        if (di == 0)
            tb.ter[sb] = static_cast<uint8_t>(er + 127);
        const int e = er + di - 3;
        uint2 m = make_uint2(0u, 0u);
        if (di < 9 && e >= -127 && e <= 126) {
            const float se = exp2_neg(e);
            const float x = __fmul_rn(P, se), y = __fmul_rn(decode(1.5f * S), se);
            const uint32_t r1 = __float_as_uint(e2m1_code_scaled<0>(__fmul_rn(decode(0.5f * S), se)));
            const uint32_t r2 = __float_as_uint(e2m1_code_scaled<0>(x));
            const uint32_t r3 = __float_as_uint(e2m1_code_scaled<0>(y));
            m = pack_code_map(r1, r2, r3, __float_as_uint(e2m1_code_scaled<1>(x)),
                              __float_as_uint(e2m1_code_scaled<1>(y)), __float_as_uint(e2m1_code_scaled<2>(x)),
                              __float_as_uint(e2m1_code_scaled<2>(y)));
            // S |g| below 2^-125 (biased exponent 2): the doublings are not
            // exact there, so the codes of magnitudes 4..7 (the map's second
            // word) come from one-by-one roundings of 2S, 3S, 4S, 6S (times |g|)
            if (!(__fmul_rn(S, ag) >= __uint_as_float(2u << 23))) {
                const uint32_t w = e2m1x8_pack(__fmul_rn(decode(2.0f * S), se), __fmul_rn(decode(3.0f * S), se),
                                               __fmul_rn(decode(4.0f * S), se), __fmul_rn(decode(6.0f * S), se),
                                               0.0f, 0.0f, 0.0f, 0.0f);
                m.y = (w & 0xFu) | ((w << 4) & 0xF00u) | ((w << 8) & 0xF0000u) | ((w << 12) & 0xF000000u);
            }
        }
        tb.map[i] = m;
    }
}

// Largest magnitude code of each half of a block (words w0,w1 and w2,w3 as
// magnitude-only nibbles m0..m3, with m0h..m3h = m >> 16): a byte-permute
// one-hot lookup turns every nibble into bit (1 << m); the OR over a half is
// the set of magnitudes present and its top bit the largest code.
__device__ __forceinline__ void max_codes(uint32_t m0, uint32_t m0h, uint32_t m1, uint32_t m1h, uint32_t m2,
                                          uint32_t m2h, uint32_t m3, uint32_t m3h, uint32_t& mm0, uint32_t& mm1)
{
    constexpr uint32_t kLo = 0x08040201u, kHi = 0x80402010u;
    const uint32_t p0 = __byte_perm(kLo, kHi, m0) | __byte_perm(kLo, kHi, m0h) | __byte_perm(kLo, kHi, m1) |
                        __byte_perm(kLo, kHi, m1h);
    const uint32_t p1 = __byte_perm(kLo, kHi, m2) | __byte_perm(kLo, kHi, m2h) | __byte_perm(kLo, kHi, m3) |
                        __byte_perm(kLo, kHi, m3h);
    // fold 4 bytes of each half: z = [p0.b0|p0.b2, p1.b0|p1.b2, p0.b1|p0.b3, p1.b1|p1.b3]
    const uint32_t z = __byte_perm(p0, p1, 0x5140u) | __byte_perm(p0, p1, 0x7362u);
    const uint32_t w = z | (z >> 16);
    mm0 = 31u - __clz((w & 0xFFu) | 1u);
    mm1 = 31u - __clz(((w >> 8) & 0xFFu) | 1u);
}

// Applies a magnitude map to the 8 codes of one word (m = magnitudes, mh =
// m >> 16): the map's bytes for nibbles 0..3 and 4..7 are regrouped into the
// even and the odd nibbles and packed with one multiply-add; the sign bits
// come from ws (the input word with its signs flipped where the scale times
// g is negative).
__device__ __forceinline__ uint32_t apply_map(uint32_t ws, uint32_t m, uint32_t mh, uint2 t)
{
    const uint32_t lo = __byte_perm(t.x, t.y, m);
    const uint32_t hi = __byte_perm(t.x, t.y, mh);
    const uint32_t ev = __byte_perm(lo, hi, 0x6420u);  // codes of nibbles 0, 2, 4, 6
    const uint32_t od = __byte_perm(lo, hi, 0x7531u);  // codes of nibbles 1, 3, 5, 7
    return (od * 16u + ev) | (ws & 0x88888888u);
}

// One block: codes in 4 words, its two E4M3 scale bytes in the low 16 bits of
// `sc` (low byte = elements 0..15).  Returns the scale byte; writes the 4
// output words.  kFlip: some scale byte of the warp's blocks is negative or
// g < 0 (otherwise every element keeps the sign of its code).
template <bool kFlip>
__device__ __forceinline__ uint32_t requant_block(const uint32_t* w, uint32_t sc, uint32_t gsign,
                                                  const RequantTables& tb, uint32_t* out)
{
    const uint32_t s0 = sc & 0x7Fu, s1 = (sc >> 8) & 0x7Fu;
    const uint32_t m0 = w[0] & 0x77777777u, m1 = w[1] & 0x77777777u;
    const uint32_t m2 = w[2] & 0x77777777u, m3 = w[3] & 0x77777777u;
    const uint32_t m0h = m0 >> 16, m1h = m1 >> 16, m2h = m2 >> 16, m3h = m3 >> 16;
    uint32_t mm0, mm1;
    max_codes(m0, m0h, m1, m1h, m2, m2h, m3, m3h, mm0, mm1);
    const int eb = max(tb.texp[s0 * 8 + mm0], tb.texp[s1 * 8 + mm1]);  // e + 127
    if (eb == 255) {  // NaN or Inf somewhere in the block
        out[0] = out[1] = out[2] = out[3] = 0u;
        return 0xFFu;
    }
    // entry d + 3 = e - er + 3 = (e + 127) + 3 - biased exponent of RN(S |g|).
    // It is >= 0 for a half with a nonzero code; an all-zero half maps to 0
    // from any entry, so a negative value (wrapping around as unsigned) and
    // values past the last entry both take entry 9.
    const uint32_t i0 = min(static_cast<uint32_t>(eb + 3 - static_cast<int>(tb.ter[s0])), uint32_t(kMapD - 1));
    const uint32_t i1 = min(static_cast<uint32_t>(eb + 3 - static_cast<int>(tb.ter[s1])), uint32_t(kMapD - 1));
    const uint2 t0 = tb.map[s0 * kMapD + i0];
    const uint2 t1 = tb.map[s1 * kMapD + i1];
    uint32_t w0 = w[0], w1 = w[1], w2 = w[2], w3 = w[3];
    if constexpr (kFlip) {
        // element sign = code sign ^ scale sign ^ sign of g
        const uint32_t f0 = (((sc >> 7) ^ gsign) & 1u) * 0x88888888u;
        const uint32_t f1 = (((sc >> 15) ^ gsign) & 1u) * 0x88888888u;
        w0 ^= f0;
        w1 ^= f0;
        w2 ^= f1;
        w3 ^= f1;
    }
    out[0] = apply_map(w0, m0, m0h, t0);
    out[1] = apply_map(w1, m1, m1h, t0);
    out[2] = apply_map(w2, m2, m2h, t1);
    out[3] = apply_map(w3, m3, m3h, t1);
    return static_cast<uint32_t>(eb);
}

struct RequantLane {
    uint32_t w[16];  // 4 blocks x 4 code words
    uint32_t sc[4];  // per block: its two E4M3 bytes
};

// Loads a lane's blocks c0 .. c0 + nreal - 1 of a row (16-byte code
// accesses, 2-byte scale accesses: any K % 32 == 0 and 16-byte alignment).
__device__ __forceinline__ void requant_lane_load(RequantLane& L, const uint8_t* __restrict__ wp,
                                                  const uint8_t* __restrict__ ws, int64_t row, int c0, int nreal,
                                                  int64_t K)
{
    const uint8_t* cp = wp + row * (K / 2) + static_cast<int64_t>(c0) * 16;
    const uint8_t* sp = ws + row * (K / 16) + static_cast<int64_t>(c0) * 2;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        uint32_t sc = 0u;
        if (j < nreal) {
            v = ld_nc_u4_cached(cp + 16 * j);
            sc = ld_stream_u16(sp + 2 * j);
        }
        L.w[4 * j] = v.x;
        L.w[4 * j + 1] = v.y;
        L.w[4 * j + 2] = v.z;
        L.w[4 * j + 3] = v.w;
        L.sc[j] = sc;
    }
}

// Row-based kernel for the shapes the flat kernel below does not take
// (K % 128 != 0 or arrays aligned to 16 bytes only).
__global__ void __launch_bounds__(kThreads) requant_kernel(const uint8_t* __restrict__ wp,
                                                           const uint8_t* __restrict__ ws, float g,
                                                           uint8_t* __restrict__ op, uint8_t* __restrict__ osf,
                                                           int64_t N, int64_t K, int64_t rows, int kb, int kbp,
                                                           int nch, int rule, int swizzled)
{
    __shared__ RequantTables tb;
    const float ag = fabsf(g);
    const uint32_t gsign = __float_as_uint(g) >> 31;
    build_code_maps(ag, rule, tb);  // needs no global memory: overlaps the previous kernel
    __syncthreads();
    grid_dependency_wait();
    launch_dependents();

    const int lane = threadIdx.x & 31;
    const int64_t n_items = rows * nch;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
    int64_t item = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
    if (item >= n_items)
        return;
    const int64_t kb4 = kbp >> 2;
    int64_t row = item / nch;
    int c0 = static_cast<int>(item - row * nch) * 128 + 4 * lane;
    int nreal = row < N ? min(max(kb - c0, 0), 4) : 0;
    RequantLane cur;
    requant_lane_load(cur, wp, ws, row, c0, nreal, K);
    while (true) {
        const int64_t next = item + stride;
        int64_t nrow = 0;
        int nc0 = 0, nnreal = 0;
        RequantLane nxt;
        if (next < n_items) {
            nrow = next / nch;
            nc0 = static_cast<int>(next - nrow * nch) * 128 + 4 * lane;
            nnreal = nrow < N ? min(max(kb - nc0, 0), 4) : 0;
            requant_lane_load(nxt, wp, ws, nrow, nc0, nnreal, K);
        }
        uint32_t out[16];
        uint32_t sfw = 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t sf = requant_block<true>(cur.w + 4 * j, cur.sc[j], gsign, tb, out + 4 * j);
            if (j < nreal)
                sfw |= sf << (8 * j);
        }
        uint8_t* dst = op + row * (K / 2) + static_cast<int64_t>(c0) * 16;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (j < nreal)
                *reinterpret_cast<uint4*>(dst + 16 * j) =
                    make_uint4(out[4 * j], out[4 * j + 1], out[4 * j + 2], out[4 * j + 3]);
        if (swizzled) {
            if (c0 < kbp)  // pad block columns and pad rows get zero bytes
                *reinterpret_cast<uint32_t*>(osf + sf_swizzled_offset(row, c0, kb4)) = sfw;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (j < nreal)
                    osf[row * kb + c0 + j] = static_cast<uint8_t>(sfw >> (8 * j));
        }
        if (next >= n_items)
            break;
        item = next;
        row = nrow;
        c0 = nc0;
        nreal = nnreal;
        cur = nxt;
    }
}

// Flat variant for K % 128 == 0 with 32-byte aligned code arrays and 8-byte
// aligned scales.  Rows are then back to back in memory and a row's block
// count is a multiple of 4, so a tensor is one run of 32-element blocks and a
// warp item is 128 consecutive blocks whatever K is (a lane's 4 blocks never
// straddle rows).  A launch covers rows [r0, r0 + n_rows) of each tensor,
// counted up to rows_pad (the 128-row padding of a swizzled scale array; pad
// rows get zero scale bytes), with every block index of that range below
// 2^32.  Grouped: E tensors of N rows stored back to back, each with its own
// global scale g[e] (device array); a run of ctas_per_e CTAs serves one
// tensor, so a CTA builds the code maps of one g only.  Dense launches use
// one 1024-thread CTA per SM (one set of code maps per SM, built by all its
// threads); grouped ones four 256-thread CTAs per SM, so that a tensor's
// CTAs spread over the SMs.  Both bounds keep a thread at 64 registers.
// Each warp walks its items two at a time from two register buffers: the
// next item's loads are in flight while the current one is converted.
struct FlatLane {
    uint32_t w[16];  // 4 blocks x 4 code words
    uint32_t s[2];   // the blocks' 8 E4M3 bytes
};

template <bool kGrouped, int kT>
__global__ void __launch_bounds__(kT, kGrouped ? 4 : 1)
    requant_flat_kernel(const uint8_t* __restrict__ wp, const uint8_t* __restrict__ ws, float g_dense,
                        const float* __restrict__ g_dev, uint8_t* __restrict__ op, uint8_t* __restrict__ osf,
                        int64_t N, int64_t K, int64_t r0, uint32_t n_rows, uint32_t rows_pad, int kb, uint32_t items,
                        int ctas_per_e, int64_t sf_e_bytes, int rule, int swizzled, DivMagic kb_div)
{
    __shared__ RequantTables tb;
    const int e = kGrouped ? static_cast<int>(blockIdx.x) / ctas_per_e : 0;
    const int local = kGrouped ? static_cast<int>(blockIdx.x) - e * ctas_per_e : static_cast<int>(blockIdx.x);
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t stride = static_cast<uint32_t>(ctas_per_e) * (kT / 32);
    uint32_t item = static_cast<uint32_t>(local) * (kT / 32) + (threadIdx.x >> 5);
    const uint32_t nreal = n_rows * static_cast<uint32_t>(kb);    // the range's real blocks come first
    const uint32_t nblocks = rows_pad * static_cast<uint32_t>(kb);  // pad rows included
    const uint32_t kb4 = static_cast<uint32_t>(kb) >> 2;
    const int64_t row0 = static_cast<int64_t>(e) * N + r0;
    const uint8_t* wpe = wp + row0 * (K / 2);
    const uint8_t* wse = ws + row0 * (K / 16);
    uint8_t* ope = op + row0 * (K / 2);
    uint8_t* osfe = osf + (swizzled ? static_cast<int64_t>(e) * sf_e_bytes : static_cast<int64_t>(e) * N * kb) + r0 * kb;

    auto load = [&](FlatLane& L, uint32_t it) {
        // the lane's first block; lanes past the range's real blocks load the
        // last real ones (their results are never stored), so the loads need
        // no branch
        const uint32_t f = min(it * 128u + 4u * lane, nreal - 4u);
        ld_nc_v8(wpe + static_cast<size_t>(f) * 16, *reinterpret_cast<uint32_t(*)[8]>(L.w));
        ld_nc_v8(wpe + static_cast<size_t>(f) * 16 + 32, *reinterpret_cast<uint32_t(*)[8]>(L.w + 8));
        const uint2 s2 = ld_nc_u64(wse + static_cast<size_t>(f) * 2);
        L.s[0] = s2.x;
        L.s[1] = s2.y;
    };

    // The first item's loads go out before the code maps are built, so that
    // building them overlaps the loads' latency.
    grid_dependency_wait();
    launch_dependents();
    FlatLane A, B;
    if (item < items)
        load(A, item);
    const float g = kGrouped ? __ldg(g_dev + e) : g_dense;
    build_code_maps(fabsf(g), rule, tb);
    __syncthreads();
    if (item >= items)
        return;
    const uint32_t gsign = __float_as_uint(g) >> 31;

    auto convert = [&](const FlatLane& L, uint32_t it) {
        const uint32_t f = it * 128u + 4u * lane;
        // signs change only where a scale byte is negative or g < 0: one vote
        // per warp item picks the path
        const bool flip = __any_sync(0xFFFFFFFFu, (gsign | ((L.s[0] | L.s[1]) & 0x80808080u)) != 0u);
        if (f >= nblocks)
            return;
        const bool real = f < nreal;
        uint32_t sfw = 0u;
        // two blocks at a time: convert, then store their 32 bytes
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t out[8];
            const uint32_t sc = L.s[h];
            if (flip) {
                sfw |= requant_block<true>(L.w + 8 * h, sc, gsign, tb, out) << (16 * h);
                sfw |= requant_block<true>(L.w + 8 * h + 4, sc >> 16, gsign, tb, out + 4) << (16 * h + 8);
            } else {
                sfw |= requant_block<false>(L.w + 8 * h, sc, 0u, tb, out) << (16 * h);
                sfw |= requant_block<false>(L.w + 8 * h + 4, sc >> 16, 0u, tb, out + 4) << (16 * h + 8);
            }
            if (real)
                st_v8(ope + static_cast<size_t>(f) * 16 + 32 * h, out);
        }
        // block index -> (row, block column) by a multiply-high
        const uint32_t row = div_by_magic(f, kb_div);
        const uint32_t c0 = f - row * static_cast<uint32_t>(kb);
        if (real) {
            if (!swizzled) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    osfe[f + j] = static_cast<uint8_t>(sfw >> (8 * j));
            }
        } else {
            sfw = 0u;  // pad rows
        }
        if (swizzled) {
            // r0 is a multiple of 128, so the range's swizzled bytes start at r0 * kb
            const uint32_t off = ((row >> 7) * kb4 + (c0 >> 2)) * 512u + (row & 31u) * 16u + ((row & 127u) >> 5) * 4u;
            *reinterpret_cast<uint32_t*>(osfe + off) = sfw;
        }
    };

    while (true) {
        const uint32_t i1 = item + stride;
        if (i1 < items)
            load(B, i1);
        convert(A, item);
        if (i1 >= items)
            break;
        const uint32_t i2 = i1 + stride;
        if (i2 < items)
            load(A, i2);
        convert(B, i1);
        if (i2 >= items)
            break;
        item = i2;
    }
}

// ------------------------------------------------------- activation quant
// (act_quant_lane and smooth_bf16x8, the MXFP4 block quantizer of one lane
// and the smooth pre-scale, live in formats.cuh: the GEMM that quantizes its
// own activations runs the same code.)

// The same block to MXFP8 (float8_e4m3fn elements) for the W4A8 fallback:
// OCP exponent e = floor(log2 amax) - 8 (8 = exponent of E4M3's largest
// value 448); the lane's 8 bytes are the nearest E4M3 values of x * 2^-e
// (ties to even, saturating at 448, sign kept), rounded two at a time by
// the hardware conversion.  q is exact in fp32 wherever it can round to a
// nonzero E4M3 value.
__device__ __forceinline__ uint2 act_quant_lane8(uint4 v, uint32_t& sf)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const uint32_t a = __vmaxu2(__vmaxu2(w[0] & 0x7FFF7FFFu, w[1] & 0x7FFF7FFFu),
                                __vmaxu2(w[2] & 0x7FFF7FFFu, w[3] & 0x7FFF7FFFu));
    uint32_t am = max(a & 0xFFFFu, a >> 16);
    am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
    am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
    const uint32_t ab = am << 16;
    if (ab >= 0x7F800000u) {
        sf = 0xFFu;
        return make_uint2(0u, 0u);
    }
    // subnormal and zero amax give <= -135, clamped to -127
    const int e = max(-127, static_cast<int>(ab >> 23) - 135);
    sf = static_cast<uint32_t>(e + 127);
    const float se = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e
    uint32_t h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float lo = __fmul_rn(__uint_as_float(w[j] << 16), se);
        const float hi = __fmul_rn(__uint_as_float(w[j] & 0xFFFF0000u), se);
        h[j] = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
    }
    return make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
}

// Smooth pre-scale preparation: float32 [K] -> bf16 [K] (nearest even) and
// a count of the values the serving path must reject (NaN, Inf, <= 0, or
// overflow / underflow to zero in bf16), added to *bad.
__global__ void __launch_bounds__(kThreads) smooth_prepare_kernel(const float* __restrict__ m,
                                                                  uint16_t* __restrict__ out, int64_t K,
                                                                  int32_t* __restrict__ bad)
{
    grid_dependency_wait();
    launch_dependents();
    int n = 0;
    for (int64_t k = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; k < K;
         k += static_cast<int64_t>(gridDim.x) * kThreads) {
        const float v = m[k];
        const __nv_bfloat16 b = __float2bfloat16_rn(v);
        const float bv = __bfloat162float(b);
        out[k] = *reinterpret_cast<const uint16_t*>(&b);
        n += (!(v > 0.0f) || isinf(v) || isinf(bv) || bv == 0.0f) ? 1 : 0;
    }
    n = __reduce_add_sync(0xFFFFFFFFu, n);
    if ((threadIdx.x & 31) == 0 && n > 0)
        atomicAdd(bad, n);
}

// Group of a grouped activation tensor whose padded scale-row range holds
// scale-row tile `tile` (group e starts at scale row 128 * the sum of
// ceil(rows_j / 128) over j < e), found by one warp on its own: a running
// prefix of the groups' tile counts, 32 groups at a time, and a ballot for
// the group whose range holds the tile.  Returns -1 past the last group;
// *first_tile is the group's first tile.  Every lane passes the same tile.
__device__ __forceinline__ int group_of_tile(const int32_t* offsets, int E, int total, int tile, int* first_tile)
{
    const int lane = threadIdx.x & 31;
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
        const int e = base + lane;
        int t = 0;
        if (e < E) {
            int start, rows;
            group_rows(offsets, e, total, &start, &rows);
            t = (rows + 127) >> 7;
        }
        int incl = t;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int n = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= d)
                incl += n;
        }
        const int first = carry + incl - t;
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, t > 0 && first <= tile && tile < first + t);
        if (hit != 0u) {
            const int src = __ffs(static_cast<int>(hit)) - 1;
            *first_tile = __shfl_sync(0xFFFFFFFFu, first, src);
            return base + src;
        }
        carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    return -1;
}

// Work item = (scale row, chunk of 8*U blocks).  For the dense tensor the
// scale row is the activation row (rows >= M are pad rows).  For the grouped
// tensor scale rows live in the padded per-group space; `grouped` selects
// the mapping.  Lane owns quarter (lane & 3) of block chunk*8U + 8u + lane/4.
// kA8: MXFP8 output (one E4M3 byte per element, rows of K bytes).
// mul (bf16 [K] or null): the smooth pre-scale; the block quantized is then
// bf16(x * mul), rounded once from the exact float32 product.
template <int U, bool kGrouped, bool kA8>
__global__ void __launch_bounds__(kThreads) act_quant_kernel(const uint16_t* __restrict__ x,
                                                             uint8_t* __restrict__ op, uint8_t* __restrict__ osf,
                                                             int64_t M, int64_t K, int64_t sf_rows, int kb,
                                                             int kbp, int nch, int uos, int swizzled,
                                                             const int32_t* __restrict__ offsets, int E,
                                                             const uint16_t* __restrict__ mul)
{
    grid_dependency_wait();
    launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t item = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t srow = item / nch;
    if (srow >= sf_rows)
        return;
    int64_t xrow = srow;
    bool row_real = srow < M;
    if (kGrouped) {
        // the group whose padded tile range holds this scale row (each warp
        // finds it itself: no block-wide prefix and barrier)
        int first_tile = 0;
        const int grp = group_of_tile(offsets, E, static_cast<int>(M), static_cast<int>(srow >> 7), &first_tile);
        if (grp < 0)
            return;
        const int64_t local = srow - static_cast<int64_t>(first_tile) * 128;
        int start_i, rows_i;
        group_rows(offsets, grp, static_cast<int>(M), &start_i, &rows_i);
        const int64_t start = start_i, rows_e = rows_i;
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
    if (mul != nullptr) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = cbase + 8 * u;
            if (c < kb)
                v[u] = smooth_bf16x8(v[u], __ldg(reinterpret_cast<const uint4*>(mul + static_cast<int64_t>(c) * 32 + q * 8)));
        }
    }
    const int64_t kb4 = kbp >> 2;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int c = cbase + 8 * u;
        const bool real = row_real && c < kb;
        uint32_t sf;
        if constexpr (kA8) {
            const uint2 codes = act_quant_lane8(v[u], sf);
            if (real)
                *reinterpret_cast<uint2*>(op + xrow * K + static_cast<int64_t>(c) * 32 + q * 8) = codes;
        } else {
            const uint32_t packed = act_quant_lane(v[u], uos, sf);
            if (real)
                *reinterpret_cast<uint32_t*>(op + xrow * (K / 2) + static_cast<int64_t>(c) * 16 + q * 4) = packed;
        }
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
// Threads walk the blocks of the scale layout: rows_pad x kbp blocks
// (swizzled: rows padded to 128 and blocks to 4, whose scale bytes are
// written as 0) or M x kb (row-major).
__global__ void __launch_bounds__(kThreads) quant_nvfp4_kernel(const uint16_t* __restrict__ x, float g,
                                                               uint8_t* __restrict__ op,
                                                               uint8_t* __restrict__ osf, int64_t halves,
                                                               int64_t M, int64_t K, int kb, int kbp, int swizzled)
{
    grid_dependency_wait();
    launch_dependents();
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    const int64_t bi = t >> 1;
    const int64_t row = bi / kbp;
    const int c = static_cast<int>(bi - row * kbp);
    // both threads of a block stay active for the shuffle
    const bool inside = t < halves;
    const bool real = inside && row < M && c < kb;
    const int64_t xoff = row * K + static_cast<int64_t>(c) * 16 + (t & 1) * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (real)
        v = ld_stream_u4(x + xoff);
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
    if (zero_codes) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t bits = (j & 1) ? (w[j >> 1] & 0xFFFF0000u) : (w[j >> 1] << 16);
            packed |= ((bits >> 28) & 0x8u) << (4 * j);
        }
    } else {
        // code = E2M1 nearest (ties to even, saturating, sign kept) of the
        // correctly rounded quotient
        float q[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t bits = (j & 1) ? (w[j >> 1] & 0xFFFF0000u) : (w[j >> 1] << 16);
            q[j] = __fdiv_rn(__uint_as_float(bits), den);
        }
        packed = e2m1x8_pack(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]);
    }
    if (real)
        *reinterpret_cast<uint32_t*>(op + xoff / 2) = packed;
    if (inside && (t & 1) == 0) {
        const uint8_t sv = real ? static_cast<uint8_t>(sb) : uint8_t(0);
        osf[swizzled ? sf_swizzled_offset(row, c, kbp >> 2) : bi] = sv;
    }
}

// ------------------------------------------------------- scale layout
// Row-major [rows][kb] scale bytes -> the swizzled layout the MMA reads,
// for either block size.  One thread per 4-byte word of the output: word w
// of 512-byte chunk (row tile rt, column group cg) holds blocks 4 cg .. +3
// of row 128 rt + 32 (w % 4) + w / 4 (pad rows and blocks as 0).
__global__ void __launch_bounds__(kThreads) sf_swizzle_kernel(const uint8_t* __restrict__ in,
                                                              uint32_t* __restrict__ out, int64_t rows, int64_t kb,
                                                              int64_t kb4, int64_t words)
{
    grid_dependency_wait();
    launch_dependents();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t wi = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; wi < words; wi += stride) {
        const int64_t chunk = wi >> 7;
        const int within = static_cast<int>(wi & 127);
        const int64_t rt = chunk / kb4;
        const int64_t c0 = (chunk - rt * kb4) * 4;
        const int64_t r = rt * 128 + (within & 3) * 32 + (within >> 2);
        uint32_t v = 0u;
        if (r < rows) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (c0 + j < kb)
                    v |= static_cast<uint32_t>(__ldg(in + r * kb + c0 + j)) << (8 * j);
        }
        out[wi] = v;
    }
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// CTAs of `kern` that fit on the whole GPU at once (per device, cached).
template <typename Kern>
int64_t resident_ctas(Kern kern, int threads = kThreads)
{
    static std::mutex mu;
    static int64_t cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 1 << 20;
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] == 0) {
        int sms = 0, per_sm = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0);
        cached[dev] = std::max<int64_t>(1, static_cast<int64_t>(sms) * std::max(per_sm, 1));
    }
    return cached[dev];
}

}  // namespace

// ------------------------------------------------------------- launchers
bool requant_flat_ok(const uint8_t* wp, const uint8_t* ws, const uint8_t* op, const uint8_t* osf, int64_t K,
                     int swizzled)
{
    return K % 128 == 0 && K < (int64_t(1) << 29) && (reinterpret_cast<uintptr_t>(wp) & 31u) == 0 && (reinterpret_cast<uintptr_t>(op) & 31u) == 0 &&
           (reinterpret_cast<uintptr_t>(ws) & 7u) == 0 && (!swizzled || (reinterpret_cast<uintptr_t>(osf) & 3u) == 0);
}

// Flat kernel over E tensors (E = 1: dense, g_dev unused), in row ranges
// whose block indices fit 32 bits (one range unless a tensor has 2^31
// blocks or more).
cudaError_t launch_requant_flat(const uint8_t* wp, const uint8_t* ws, float g, const float* g_dev, uint8_t* op,
                                uint8_t* osf, int E, int64_t N, int64_t K, int rule, int swizzled, cudaStream_t stream)
{
    constexpr int kDenseT = 1024, kGroupT = 256;
    const int kb = static_cast<int>(K / 32);
    const int64_t rows_pad = swizzled ? ceil_div(N, 128) * 128 : N;
    const int64_t sf_e_bytes = rows_pad * kb;  // swizzled bytes per tensor (kb % 4 == 0)
    // rows per launch: a multiple of 128 with at most 2^31 blocks
    const int64_t chunk = std::max<int64_t>(128, ((int64_t(1) << 31) / kb) / 128 * 128);
    const DivMagic kb_div = div_magic(static_cast<uint32_t>(kb));
    for (int64_t r0 = 0; r0 < rows_pad; r0 += chunk) {
        const int64_t pad = std::min(chunk, rows_pad - r0);
        const int64_t real = std::max<int64_t>(0, std::min(chunk, N - r0));
        const int64_t items = ceil_div(pad * kb, 128);  // warp items per tensor and launch
        cudaError_t err;
        if (g_dev == nullptr) {
            const int64_t want = ceil_div(items * 32, kDenseT);  // CTAs that give every warp one item
            const int64_t blocks = std::min<int64_t>(want, resident_ctas(requant_flat_kernel<false, kDenseT>, kDenseT));
            err = launch_pdl(requant_flat_kernel<false, kDenseT>, dim3(static_cast<unsigned>(blocks)), dim3(kDenseT),
                             0, stream, wp, ws, g, static_cast<const float*>(nullptr), op, osf, N, K, r0,
                             static_cast<uint32_t>(real), static_cast<uint32_t>(pad), kb,
                             static_cast<uint32_t>(items), static_cast<int>(blocks), sf_e_bytes, rule, swizzled,
                             kb_div);
        } else {
            const int64_t want = ceil_div(items * 32, kGroupT);
            const int64_t per_e = std::max<int64_t>(
                1, std::min<int64_t>(want, resident_ctas(requant_flat_kernel<true, kGroupT>, kGroupT) / E));
            err = launch_pdl(requant_flat_kernel<true, kGroupT>, dim3(static_cast<unsigned>(per_e * E)),
                             dim3(kGroupT), 0, stream, wp, ws, 0.0f, g_dev, op, osf, N, K, r0,
                             static_cast<uint32_t>(real), static_cast<uint32_t>(pad), kb,
                             static_cast<uint32_t>(items), static_cast<int>(per_e), sf_e_bytes, rule, swizzled,
                             kb_div);
        }
        if (err != cudaSuccess)
            return err;
    }
    return cudaSuccess;
}

// rule bits for the code maps: the block rule and the decoded-value precision
static int requant_rule(int alg, int bf16)
{
    return (alg == 2 ? kRuleUos : 0) | (bf16 ? kRuleBf16 : 0);
}

cudaError_t launch_requant(const uint8_t* wp, const uint8_t* ws, float g, uint8_t* op, uint8_t* osf, int64_t N,
                           int64_t K, int alg, int swizzled, int bf16, cudaStream_t stream)
{
    const int kb = static_cast<int>(K / 32);
    const int kbp = swizzled ? static_cast<int>(ceil_div(kb, 4) * 4) : kb;
    const int64_t rows = swizzled ? ceil_div(N, 128) * 128 : N;
    const int nch = static_cast<int>(ceil_div(kbp, 128));
    const int64_t warps = rows * nch;
    const int rule = requant_rule(alg, bf16);
    if (requant_flat_ok(wp, ws, op, osf, K, swizzled)) {
        return launch_requant_flat(wp, ws, g, nullptr, op, osf, 1, N, K, rule, swizzled, stream);
    } else {
        const int64_t blocks =
            std::min<int64_t>(ceil_div(warps * 32, kThreads), resident_ctas(requant_kernel));
        return launch_pdl(requant_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, stream, wp,
                          ws, g, op, osf, N, K, rows, kb, kbp, nch, rule, swizzled);
    }
    return cudaGetLastError();
}

cudaError_t launch_requant_grouped(const uint8_t* wp, const uint8_t* ws, const float* g_dev, uint8_t* op,
                                   uint8_t* osf, int E, int64_t N, int64_t K, int alg, int swizzled, int bf16,
                                   cudaStream_t stream)
{
    return launch_requant_flat(wp, ws, 0.0f, g_dev, op, osf, E, N, K, requant_rule(alg, bf16), swizzled, stream);
}

cudaError_t launch_act_quant(const void* x, uint8_t* op, uint8_t* osf, int64_t M, int64_t K, int alg,
                             int swizzled, cudaStream_t stream, const void* mul)
{
    constexpr int U = 4;
    const int kb = static_cast<int>(K / 32);
    const int kbp = swizzled ? static_cast<int>(ceil_div(kb, 4) * 4) : kb;
    const int64_t rows = swizzled ? ceil_div(M, 128) * 128 : M;
    const int nch = static_cast<int>(ceil_div(kbp, 8 * U));
    const int64_t blocks = ceil_div(rows * nch * 32, kThreads);
    if (blocks == 0)
        return cudaSuccess;
    return launch_pdl(act_quant_kernel<U, false, false>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0,
                      stream, static_cast<const uint16_t*>(x), op, osf, M, K, rows, kb, kbp, nch, alg == 2 ? 1 : 0,
                      swizzled, static_cast<const int32_t*>(nullptr), 0, static_cast<const uint16_t*>(mul));
}

cudaError_t launch_act_quant_mxfp8(const void* x, uint8_t* op, uint8_t* osf, int64_t M, int64_t K, int swizzled,
                                   cudaStream_t stream, const void* mul)
{
    constexpr int U = 4;
    const int kb = static_cast<int>(K / 32);
    const int kbp = swizzled ? static_cast<int>(ceil_div(kb, 4) * 4) : kb;
    const int64_t rows = swizzled ? ceil_div(M, 128) * 128 : M;
    const int nch = static_cast<int>(ceil_div(kbp, 8 * U));
    const int64_t blocks = ceil_div(rows * nch * 32, kThreads);
    if (blocks == 0)
        return cudaSuccess;
    return launch_pdl(act_quant_kernel<U, false, true>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0,
                      stream, static_cast<const uint16_t*>(x), op, osf, M, K, rows, kb, kbp, nch, 0, swizzled,
                      static_cast<const int32_t*>(nullptr), 0, static_cast<const uint16_t*>(mul));
}

cudaError_t launch_smooth_prepare(const float* m, void* out, int64_t K, int32_t* bad, cudaStream_t stream)
{
    cudaError_t err = cudaMemsetAsync(bad, 0, sizeof(int32_t), stream);
    if (err != cudaSuccess)
        return err;
    const int64_t blocks = std::min<int64_t>(ceil_div(K, kThreads), resident_ctas(smooth_prepare_kernel));
    return launch_pdl(smooth_prepare_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, stream, m,
                      static_cast<uint16_t*>(out), K, bad);
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
    return launch_pdl(act_quant_kernel<U, true, false>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, stream,
                      static_cast<const uint16_t*>(x), op, osf, total_M, K, rows, kb, kbp, nch, alg == 2 ? 1 : 0, 1,
                      offsets, E, static_cast<const uint16_t*>(nullptr));
}

cudaError_t launch_quant_nvfp4(const void* x, float g, uint8_t* op, uint8_t* osf, int64_t M, int64_t K,
                               int swizzled, cudaStream_t stream)
{
    const int kb = static_cast<int>(K / 16);
    const int kbp = swizzled ? static_cast<int>(ceil_div(kb, 4) * 4) : kb;
    const int64_t rows = swizzled ? ceil_div(M, 128) * 128 : M;
    const int64_t halves = rows * kbp * 2;
    const int64_t blocks = ceil_div(halves, kThreads);
    if (blocks == 0)
        return cudaSuccess;
    return launch_pdl(quant_nvfp4_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, stream,
                      static_cast<const uint16_t*>(x), g, op, osf, halves, M, K, kb, kbp, swizzled);
}

// ------------------------------------------------ DualScale quantization
// Online dual-level quantization of a bf16 weight ("W4A4 MXFP4
// Quantization", mxfp4_dualscale Online Mode; reading): per row and
// 512-element group, coarse = amax / 6 over the group's finite magnitudes
// (1 when there is none above zero), then the OCP MX block rule on
// y = w / coarse per 32 elements.  Both divisions are IEEE float32.  One warp
// per (row, group); lane i holds elements 16i .. 16i + 15, a lane pair one
// 32-element block.  Rows past N (the 128-row padding of a swizzled scale
// array) get zero fine bytes.
__global__ void __launch_bounds__(kThreads) dual_quant_kernel(const uint16_t* __restrict__ w, uint8_t* __restrict__ op,
                                                              uint8_t* __restrict__ ofine, float* __restrict__ ocoarse,
                                                              int64_t N, int64_t K, int64_t rows, int swizzled)
{
    grid_dependency_wait();
    launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t item = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t groups = K / 512;
    const int64_t row = item / groups;
    if (row >= rows)
        return;
    const int64_t g = item - row * groups;
    const int kb = static_cast<int>(K / 32);
    const int64_t kb4 = kb >> 2;
    const int blk = static_cast<int>(g) * 16 + (lane >> 1);  // this lane's 32-element block
    uint32_t sf = 0u;
    if (row < N) {
        const uint16_t* src = w + row * K + g * 512 + lane * 16;
        const uint4 a = ld_stream_u4(src), b = ld_stream_u4(src + 8);
        const uint32_t x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        // largest finite magnitude of the group (bf16 patterns below Inf order as their values)
        uint32_t m = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t lo = x[i] & 0x7FFFu, hi = (x[i] >> 16) & 0x7FFFu;
            m = max(m, lo < 0x7F80u ? lo : 0u);
            m = max(m, hi < 0x7F80u ? hi : 0u);
        }
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1)
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, d));
        const float amax = __uint_as_float(m << 16);
        const float coarse = amax > 0.0f ? __fdiv_rn(amax, 6.0f) : 1.0f;
        float y[16];
        uint32_t ya = 0u;  // largest |y| bits of this lane's half block (NaN / Inf above every finite)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            y[2 * i] = __fdiv_rn(__uint_as_float(x[i] << 16), coarse);
            y[2 * i + 1] = __fdiv_rn(__uint_as_float(x[i] & 0xFFFF0000u), coarse);
            ya = max(ya, __float_as_uint(y[2 * i]) & 0x7FFFFFFFu);
            ya = max(ya, __float_as_uint(y[2 * i + 1]) & 0x7FFFFFFFu);
        }
        ya = max(ya, __shfl_xor_sync(0xFFFFFFFFu, ya, 1));
        uint2 codes = make_uint2(0u, 0u);
        if (ya >= 0x7F800000u) {
            sf = 0xFFu;  // NaN or Inf in the block: scale 0xFF, zero codes
        } else {
            const int e = mx_shared_exp(ya, 0);
            sf = static_cast<uint32_t>(e + 127);
            const float se = exp2_neg(e);
#pragma unroll
            for (int i = 0; i < 16; ++i)
                y[i] = __fmul_rn(y[i], se);
            codes.x = e2m1x8_pack(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
            codes.y = e2m1x8_pack(y[8], y[9], y[10], y[11], y[12], y[13], y[14], y[15]);
        }
        *reinterpret_cast<uint2*>(op + row * (K / 2) + g * 256 + lane * 8) = codes;
        if (lane == 0)
            ocoarse[row * groups + g] = coarse;
    }
    if (swizzled) {
        // lane 8i writes the word of blocks 4i .. 4i + 3 (held by lanes 8i, 8i+2, 8i+4, 8i+6)
        const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, sf, 2);
        const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, sf, 4);
        const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, sf, 6);
        if ((lane & 7) == 0)
            *reinterpret_cast<uint32_t*>(ofine + sf_swizzled_offset(row, blk, kb4)) = sf | (b1 << 8) | (b2 << 16) | (b3 << 24);
    } else if (row < N && (lane & 1) == 0) {
        ofine[row * kb + blk] = static_cast<uint8_t>(sf);
    }
}

cudaError_t launch_dual_quant(const void* w, uint8_t* op, uint8_t* ofine, float* ocoarse, int64_t N, int64_t K,
                              int swizzled, cudaStream_t stream)
{
    const int64_t rows = swizzled ? ceil_div(N, 128) * 128 : N;
    const int64_t warps = rows * (K / 512);
    const int64_t blocks = ceil_div(warps * 32, kThreads);
    if (blocks == 0)
        return cudaSuccess;
    return launch_pdl(dual_quant_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, stream,
                      static_cast<const uint16_t*>(w), op, ofine, ocoarse, N, K, rows, swizzled);
}

cudaError_t launch_sf_swizzle(const uint8_t* in, uint8_t* out, int64_t rows, int64_t kb, cudaStream_t stream)
{
    const int64_t kb4 = ceil_div(kb, 4);
    const int64_t words = ceil_div(rows, 128) * kb4 * 128;
    const int64_t blocks = std::min<int64_t>(ceil_div(words, kThreads), resident_ctas(sf_swizzle_kernel));
    if (blocks == 0)
        return cudaSuccess;
    return launch_pdl(sf_swizzle_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, stream, in,
                      reinterpret_cast<uint32_t*>(out), rows, kb, kb4, words);
}

}  // namespace fp4lin
