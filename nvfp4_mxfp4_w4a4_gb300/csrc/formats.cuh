// formats.cuh -- device-side element codecs for the quantizers.
//
// E2M1 grid (magnitudes, code 0..7): 0, 0.5, 1, 1.5, 2, 3, 4, 6.
// MX block rule ("W4A4 MXFP4 Quantization", Single-Scale Block Scaling):
// 32 elements share one E8M0 exponent; OCP picks floor(log2 amax) - 2,
// UOS (Qmax = 7.25) the smallest e with amax <= 7.25 * 2^e; elements are
// rounded to the nearest E2M1 value ("rint", ties to even) and saturate at 6.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace fp4lin {

// x + kMagic (|x| < 2^22) leaves rint(x) (nearest, ties to even) in the low
// mantissa bits of the float sum; the low byte of the sum's bit pattern is
// that integer for 0 <= rint(x) < 256.
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23

// Nearest E2M1 magnitude code of z * 2^j (z >= 0, not NaN), returned as
// kMagic + code.  The code of a value y is the lower envelope of the three
// lines 2y (step-0.5 part of the grid), 2 + y (step-1 part) and 4 + y/2
// (step-2 part), capped at 7; rint is monotone, so it commutes with the min
// and each line is rounded on its own (the even offsets keep ties on even
// codes).  The scaling by 2^j happens inside the fused multiply-adds, so it
// is exact.
template <int J>
__device__ __forceinline__ float e2m1_code_scaled(float z)
{
    constexpr float s2 = (J == 0) ? 2.0f : (J == 1) ? 4.0f : 8.0f;
    constexpr float s1 = (J == 0) ? 1.0f : (J == 1) ? 2.0f : 4.0f;
    constexpr float s0 = (J == 0) ? 0.5f : (J == 1) ? 1.0f : 2.0f;
    const float a = __fmaf_rn(z, s2, kMagic);
    const float b = __fmaf_rn(z, s1, kMagic + 2.0f);
    const float c = __fmaf_rn(z, s0, kMagic + 4.0f);
    return fminf(fminf(a, b), fminf(c, kMagic + 7.0f));
}

__device__ __forceinline__ uint32_t e2m1_code(float z)
{
    return __float_as_uint(e2m1_code_scaled<0>(z)) & 0xFFu;
}

// Eight values to eight E2M1 codes in one word (value 2k in bits 8k..8k+3,
// value 2k+1 in bits 8k+4..8k+7): the hardware pair conversion, which rounds
// to the nearest grid value with ties to the even code, saturates at +-6 and
// keeps the sign of zero, as the MX encoding wants.
__device__ __forceinline__ uint32_t e2m1x8_pack(float q0, float q1, float q2, float q3, float q4, float q5, float q6,
                                                float q7)
{
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(q0), "f"(q1), "f"(q2), "f"(q3), "f"(q4), "f"(q5), "f"(q6), "f"(q7));
    return r;
}

// Shared exponent from the fp32 bit pattern of a finite, non-negative amax.
// For a normal amax = (1 + f) * 2^E the OCP exponent is E - 2 (biased field
// minus 129); UOS adds one when 1 + f > 1.8125 (mantissa field > 0x680000).
// Subnormal and zero amax give <= -128, which the clamp turns into -127.
__device__ __forceinline__ int mx_shared_exp(uint32_t amax_bits, int uos)
{
    int e = static_cast<int>(amax_bits >> 23) - 129;
    if (uos)
        e += (amax_bits & 0x7FFFFFu) > 0x680000u ? 1 : 0;
    return max(-127, min(127, e));
}

// 2^-e as a float (e in [-127, 126]).
__device__ __forceinline__ float exp2_neg(int e)
{
    return __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
}

// E2M1 value of a magnitude code 0..7 (exact float).
__device__ __forceinline__ float e2m1_mag_value(uint32_t m)
{
    if (m < 2)
        return 0.5f * static_cast<float>(m);
    return __uint_as_float((((m >> 1) + 126u) << 23) | ((m & 1u) << 22));
}

// Two float8_e4m3fn bytes (low byte first) -> two floats, exactly.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_bytes)
{
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_bytes & 0xFFFFu),
                                                     __NV_E4M3);
    return make_float2(__half2float(__ushort_as_half(h.x)), __half2float(__ushort_as_half(h.y)));
}

// float -> float8_e4m3fn, round to nearest even, saturating to +-448, NaN -> 0x7F.
__device__ __forceinline__ uint32_t float_to_e4m3_satfinite(float t)
{
    const __nv_fp8x2_storage_t v = __nv_cvt_float2_to_fp8x2(make_float2(t, t), __NV_SATFINITE, __NV_E4M3);
    return static_cast<uint32_t>(v) & 0xFFu;
}

// Exact n / d for 0 <= n < 2^32 by a divisor d fixed for a launch, by one
// multiply-high and shifts: the round-up method of Granlund and Montgomery,
// "Division by invariant integers using multiplication" (PLDI 1994),
// section 4.  With l = ceil(log2 d): m = floor(2^32 (2^l - d) / d) + 1,
// s1 = min(l, 1), s2 = max(l - 1, 0).
struct DivMagic {
    uint32_t m, s1, s2;
};

__host__ __device__ inline DivMagic div_magic(uint32_t d)
{
    uint32_t l = 0;
    while ((uint64_t(1) << l) < d)
        ++l;
    DivMagic g;
    g.m = static_cast<uint32_t>(((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1);
    g.s1 = l < 1 ? l : 1;
    g.s2 = l > 1 ? l - 1 : 0;
    return g;
}

__device__ __forceinline__ uint32_t div_by_magic(uint32_t n, DivMagic g)
{
    const uint32_t t = __umulhi(g.m, n);
    return (t + ((n - t) >> g.s1)) >> g.s2;
}

// Rows [start, start + rows) of group e from the row offsets, each offset
// clamped to [0, total] (and the end to >= the start): offsets that are out
// of order or out of range can then give wrong groups but never an access
// outside the total rows.
__device__ __forceinline__ void group_rows(const int32_t* offsets, int e, int total, int* start, int* rows)
{
    const int a = min(max(__ldg(offsets + e), 0), total);
    const int b = min(max(__ldg(offsets + e + 1), a), total);
    *start = a;
    *rows = b - a;
}

// Scale-factor byte offset of (row r, 32-block c) in the swizzled layout the
// block-scaled MMA reads; kb4 = ceil(K/32 / 4).
__device__ __forceinline__ int64_t sf_swizzled_offset(int64_t r, int64_t c, int64_t kb4)
{
    return ((r >> 7) * kb4 + (c >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (c & 3);
}


// ------------------------------------------------------- activation quant
// One lane holds 8 consecutive bf16 of a 32-element block (4 lanes per
// block).  Returns the packed codes (4 bytes) and, through `sf`, the block's
// scale byte (the same on all 4 lanes).  q = x * 2^-e is exact in fp32 (a
// bf16 value times a power of two; e <= 125 for a finite bf16 amax and
// e >= -127 after the clamp, so 2^-e is a normal fp32), and the hardware
// pair conversion rounds it to E2M1.
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
    const float se = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e
    float q[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        q[2 * j] = __fmul_rn(__uint_as_float(w[j] << 16), se);
        q[2 * j + 1] = __fmul_rn(__uint_as_float(w[j] & 0xFFFF0000u), se);
    }
    return e2m1x8_pack(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]);
}

// Eight bf16 times eight bf16, each product rounded once to bf16 (the exact
// float32 product of two bf16 values, then round to nearest even).
__device__ __forceinline__ uint4 smooth_bf16x8(uint4 x, uint4 m)
{
    const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
    const uint32_t mw[4] = {m.x, m.y, m.z, m.w};
    uint32_t r[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float lo = __fmul_rn(__uint_as_float(xw[j] << 16), __uint_as_float(mw[j] << 16));
        const float hi = __fmul_rn(__uint_as_float(xw[j] & 0xFFFF0000u), __uint_as_float(mw[j] & 0xFFFF0000u));
        const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
        r[j] = *reinterpret_cast<const uint32_t*>(&b);
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
}

}  // namespace fp4lin
