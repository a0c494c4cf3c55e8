// Static FP8 (e4m3) quantisation of storage values for the LayerNorm +
// modulate output pass: e4m3(RN(y / qs)), round to nearest even, saturating
// at +-448, NaN to NaN; the quotient is exact without a division per value.
#pragma once
#include <cuda_fp8.h>

#include "common.cuh"

namespace adaln {

// a / b rounded to nearest even, from r = RN(1/b): Markstein's correction
// (P. Markstein, IBM J. Res. Dev. 34(1), 1990; the Handbook of
// Floating-Point Arithmetic's FMA-based division): q = RN(a r); the residual
// e = a - q b is exact through one FMA; q' = RN(q + e r) is RN(a / b) when
// neither the residual nor the product leaves the range where they are
// exact.  With |a| and |q| in [2^-100, 2^100] the residual's lowest bit is
// at least 2^-147, so it is exact even when subnormal; outside that range
// (zeros, tiny, huge, infinite, NaN) the quotient comes from __fdiv_rn.
__device__ __forceinline__ float div_by_recip(float a, float b, float r) {
    const float q = __fmul_rn(a, r);
    const float mq = fabsf(q), ma = fabsf(a);
    if (!(mq >= 0x1p-100f && mq <= 0x1p+100f && ma >= 0x1p-100f && ma <= 0x1p+100f)) return __fdiv_rn(a, b);
    const float e = __fmaf_rn(-q, b, a);
    return __fmaf_rn(e, r, q);
}

// Static FP8 quantisation: e4m3(RN(y / qs)) of storage values y, round to
// nearest even, saturating.  With qr = RN(1 / qs), Markstein's correction
// (div_by_recip) is exact when |y| and |y / qs| lie in [2^-100, 2^100]; the
// kernel turns that into a window [lo, hi] of 16-bit magnitude patterns
// (|y| >= max(2^-100, 2^-99 / |qr|), |y| <= min(2^100, 2^99 / |qr|): a
// factor 2 of margin for the product's rounding), checks a chunk's 4
// magnitudes against it with one packed min, one max and two compares,
// runs the correction on f32x2 pairs when they all fit, and takes the exact
// quotient one value at a time (zeros, NaN, extreme magnitudes) otherwise.
//
// For an ordinary positive scale (2^-60 <= qs <= 2^60, and the window's
// upper bound at least 1024 qs) a branch-free form (quant4_e4m3_fast) gives
// the same codes: each value's magnitude is clamped to the window's upper
// bound (every |y| above it saturates to 448 either way) and its sign flipped
// in one packed min.NaN.xorsign.abs with the negated bound, and the
// correction runs on -y:
// q = RN(y r), e' = RN(q qs - y) = -e, q' = RN(q - e' r), the same values as
// above, but with zeros that keep their sign (RN(q + e r) turns -0 into +0).
// Below the window's lower bound the correction may be inexact, but there
// |y / qs| < 2^-40: the code is a signed zero either way, and the sign comes
// out right (q is RN(y r) or carries its sign).  Infinities become the
// clamped bound (saturating), NaN stays NaN.
struct QuantE4M3 {
    float qs, qr, nqs;  // the scale, RN(1 / scale), -scale
    uint32_t lo2, hi2;  // the pattern window, in both 16-bit halves
    uint32_t nhi2;      // the upper bound's pattern with the sign bit set, in both halves
    bool fast;          // the scale is ordinary and positive: quant4_e4m3_fast applies
};

template <DT T> __device__ __forceinline__ uint32_t pattern_ceil(float t);
template <DT T> __device__ __forceinline__ uint32_t pattern_floor(float t);
template <> __device__ __forceinline__ uint32_t pattern_ceil<DT::BF16>(float t) {
    return (__float_as_uint(t) + 0xffffu) >> 16;  // t > 0 finite
}
template <> __device__ __forceinline__ uint32_t pattern_floor<DT::BF16>(float t) { return __float_as_uint(t) >> 16; }
template <> __device__ __forceinline__ uint32_t pattern_ceil<DT::FP16>(float t) {
    return __half_as_ushort(__float2half_ru(t));
}
template <> __device__ __forceinline__ uint32_t pattern_floor<DT::FP16>(float t) {
    return __half_as_ushort(__float2half_rd(t));
}
template <DT T> __device__ __forceinline__ float pattern_value(uint32_t p);
template <> __device__ __forceinline__ float pattern_value<DT::BF16>(uint32_t p) { return __uint_as_float(p << 16); }
template <> __device__ __forceinline__ float pattern_value<DT::FP16>(uint32_t p) {
    return __half2float(__ushort_as_half((unsigned short)p));
}

template <DT T>
__device__ __forceinline__ QuantE4M3 quant_setup(float qs) {
    QuantE4M3 c;
    c.qs = qs;
    c.qr = __frcp_rn(qs);
    c.nqs = -qs;
    const float ar = fabsf(c.qr);
    const float lo = fmaxf(0x1p-100f, __fdiv_rn(0x1p-99f, ar));
    const float hi = fminf(0x1p+100f, __fdiv_rn(0x1p+99f, ar));
    uint32_t lp = 0xffffu, hp = 0u;  // empty window (every chunk exact) unless the bounds are ordinary
    if (lo <= hi && lo > 0.0f && hi < 0x1p+101f) {
        lp = pattern_ceil<T>(lo);
        hp = pattern_floor<T>(hi);
    }
    c.lo2 = lp | (lp << 16);
    c.hi2 = hp | (hp << 16);
    // (false for NaN and every negative scale; an fp16 bound of 65504 needs qs <= 63.97)
    c.fast = qs >= 0x1p-60f && qs <= 0x1p+60f && pattern_value<T>(hp) >= 1024.0f * qs;
    const uint32_t nh = (c.fast ? hp : 0u) | 0x8000u;
    c.nhi2 = nh | (nh << 16);
    return c;
}

// (by value: the values stay in registers; the call is rare)
static __device__ __noinline__ float4 quant_exact4(float4 a, float qs, float qr) {
    return make_float4(div_by_recip(a.x, qs, qr), div_by_recip(a.y, qs, qr), div_by_recip(a.z, qs, qr),
                       div_by_recip(a.w, qs, qr));
}

// every |value| of the two packed pairs lies in [lo, hi] (lo2 / hi2: the
// bounds' patterns in both halves); the storage type's own packed min / max
// and compares, on magnitudes (a NaN may pass: its quotient is NaN either way)
template <DT T> __device__ __forceinline__ bool window4(uint32_t m0, uint32_t m1, uint32_t lo2, uint32_t hi2);
template <> __device__ __forceinline__ bool window4<DT::BF16>(uint32_t m0, uint32_t m1, uint32_t lo2, uint32_t hi2) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&m0);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&m1);
    return __hble2(__hmax2(a, b), *reinterpret_cast<const __nv_bfloat162 *>(&hi2)) &&
           __hbge2(__hmin2(a, b), *reinterpret_cast<const __nv_bfloat162 *>(&lo2));
}
template <> __device__ __forceinline__ bool window4<DT::FP16>(uint32_t m0, uint32_t m1, uint32_t lo2, uint32_t hi2) {
    const __half2 a = *reinterpret_cast<const __half2 *>(&m0);
    const __half2 b = *reinterpret_cast<const __half2 *>(&m1);
    return __hble2(__hmax2(a, b), *reinterpret_cast<const __half2 *>(&hi2)) &&
           __hbge2(__hmin2(a, b), *reinterpret_cast<const __half2 *>(&lo2));
}

// -clamp(y) of a packed pair: min(|y|, |b|) with the sign of y flipped (b
// negative), NaN kept
template <DT T> __device__ __forceinline__ uint32_t neg_clamp16x2(uint32_t y, uint32_t nb);
template <> __device__ __forceinline__ uint32_t neg_clamp16x2<DT::BF16>(uint32_t y, uint32_t nb) {
    uint32_t r;
    asm("min.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(y), "r"(nb));
    return r;
}
template <> __device__ __forceinline__ uint32_t neg_clamp16x2<DT::FP16>(uint32_t y, uint32_t nb) {
    uint32_t r;
    asm("min.NaN.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(r) : "r"(y), "r"(nb));
    return r;
}

// the e4m3 codes of 4 storage values (2 packed pairs), in memory order, for
// an ordinary positive scale (c.fast): no branch
template <DT T>
__device__ __forceinline__ uint32_t quant4_e4m3_fast(const uint32_t *o, const QuantE4M3 &c) {
    const uint32_t n0 = neg_clamp16x2<T>(o[0], c.nhi2), n1 = neg_clamp16x2<T>(o[1], c.nhi2);
    const f2_t a01 = f2(lo_f32<T>(n0), hi_f32<T>(n0)), a23 = f2(lo_f32<T>(n1), hi_f32<T>(n1));  // -y
    const f2_t nr2 = f2(-c.qr, -c.qr), s2 = f2(c.qs, c.qs);
    f2_t p01 = f2_mul(a01, nr2), p23 = f2_mul(a23, nr2);  // RN(y r)
    p01 = f2_fma(f2_fma(p01, s2, a01), nr2, p01);         // q - (q s - y) r
    p23 = f2_fma(f2_fma(p23, s2, a23), nr2, p23);
    float q0, q1, q2, q3;
    f2_split(p01, q0, q1);
    f2_split(p23, q2, q3);
    const uint32_t q01 = __nv_cvt_float2_to_fp8x2(make_float2(q0, q1), __NV_SATFINITE, __NV_E4M3);
    const uint32_t q23 = __nv_cvt_float2_to_fp8x2(make_float2(q2, q3), __NV_SATFINITE, __NV_E4M3);
    return (q01 & 0xffffu) | (q23 << 16);
}

// the e4m3 codes of 4 storage values (2 packed pairs), in memory order, for
// any scale: the window check, the correction, the exact quotient outside
template <DT T>
__device__ __forceinline__ uint32_t quant4_e4m3_window(const uint32_t *o, const QuantE4M3 &c) {
    float q0, q1, q2, q3;
    if (window4<T>(o[0] & 0x7fff7fffu, o[1] & 0x7fff7fffu, c.lo2, c.hi2)) {
        const f2_t a01 = f2(lo_f32<T>(o[0]), hi_f32<T>(o[0])), a23 = f2(lo_f32<T>(o[1]), hi_f32<T>(o[1]));
        const f2_t r2 = f2(c.qr, c.qr), nb2 = f2(c.nqs, c.nqs);
        f2_t p01 = f2_mul(a01, r2), p23 = f2_mul(a23, r2);
        p01 = f2_fma(f2_fma(p01, nb2, a01), r2, p01);  // q + (a - q b) r
        p23 = f2_fma(f2_fma(p23, nb2, a23), r2, p23);
        f2_split(p01, q0, q1);
        f2_split(p23, q2, q3);
    } else {
        const float4 e = quant_exact4(make_float4(lo_f32<T>(o[0]), hi_f32<T>(o[0]), lo_f32<T>(o[1]), hi_f32<T>(o[1])),
                                      c.qs, c.qr);
        q0 = e.x;
        q1 = e.y;
        q2 = e.z;
        q3 = e.w;
    }
    const uint32_t q01 = __nv_cvt_float2_to_fp8x2(make_float2(q0, q1), __NV_SATFINITE, __NV_E4M3);
    const uint32_t q23 = __nv_cvt_float2_to_fp8x2(make_float2(q2, q3), __NV_SATFINITE, __NV_E4M3);
    return (q01 & 0xffffu) | (q23 << 16);
}

template <DT T>
__device__ __forceinline__ uint32_t quant4_e4m3(const uint32_t *o, const QuantE4M3 &c) {
    return c.fast ? quant4_e4m3_fast<T>(o, c) : quant4_e4m3_window<T>(o, c);
}

}  // namespace adaln
