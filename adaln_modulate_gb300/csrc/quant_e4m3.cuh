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
//
// Cheaper still (quant4_e4m3_plain): the code of the product RN(y p) alone,
// for a multiplier p near 1 / qs whose codes equal those of RN(y / qs) for
// every storage value.  For y = M 2^E (M the significand; a subnormal
// normalises to one of the same M) the two are the scaled values
// RN(M p) 2^E and RN(M / qs) 2^E, so it is enough to compare the two codes
// for every significand M (128 for bf16, 1024 for fp16) and every E that
// puts the quotient in [2^-12, 2^11): below that both codes are signed
// zeros, above both are +-448.  Zeros, infinities and NaN need nothing
// (RN(y p) is a signed zero, +-inf, NaN).  The check (quant_plain_share) is
// run once per CTA, split over its threads, for p = r, then r -+ 1 ulp and
// r -+ 2 ulp (quant_pick_plain); r itself fails when some quotient lies
// within an ulp of an e4m3 rounding boundary, and every p fails for exact
// ties (y = m s with m a midpoint) that the product rounds the other way.
struct QuantE4M3 {
    float qs, qr, nqs;  // the scale, RN(1 / scale), -scale
    uint32_t lo2, hi2;  // the pattern window, in both 16-bit halves
    uint32_t nhi2;      // the upper bound's pattern with the sign bit set, in both halves
    bool fast;          // the scale is ordinary and positive: quant4_e4m3_fast applies
    bool plain;         // quant4_e4m3_plain applies, with the multiplier rp (quant_pick_plain)
    float rp;
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
    c.plain = false;
    c.rp = c.qr;
    return c;
}

// q 2^j for a normal q whose product stays normal (exact)
__device__ __forceinline__ float scale_pow2(float q, int j) {
    return __uint_as_float(__float_as_uint(q) + ((uint32_t)j << 23));
}

// The multiplier candidate t of the plain-product search: r, r - 1 ulp,
// r + 1 ulp, r - 2 ulp, r + 2 ulp (r > 0)
constexpr int kPlainTries = 5;
__device__ __forceinline__ float plain_candidate(float r, int t) {
    const int k = ((t + 1) >> 1) * ((t & 1) ? -1 : 1);
    return __uint_as_float(__float_as_uint(r) + (uint32_t)k);
}

// One thread's share of the plain-product check for the multiplier p:
// significands M = 1 + i 2^-F (F = 7 for bf16, 10 for fp16), i = first,
// first + stride, ...  True when, for each of them, RN(M p) 2^j and
// RN(M / qs) 2^j have the same code for every j that puts RN(M / qs) 2^j in
// [2^-12, 2^11).  The code of a value depends on its binade only through the
// number of significand bits e4m3 keeps there: the binades [2^-11, 2^-10)
// .. [2^-7, 2^-6) each keep their own number (zero threshold, subnormals),
// the normal ones [2^-6, 2^8) all keep three and [2^8, 2^9) three with the
// saturation at 448, so one binade stands for all the normal ones.  Near a
// binade boundary both values round to the boundary's code.  With
// 2^-60 <= qs <= 2^60 every value involved is a normal binary32.
template <DT T>
__device__ __forceinline__ bool quant_plain_share(const QuantE4M3 &c, float p, int first, int stride) {
    constexpr int F = T == DT::BF16 ? 7 : 10;
    constexpr int kBinades[7] = {-11, -10, -9, -8, -7, 0, 8};
    if (!c.fast) return false;
    bool ok = true;
    for (int i = first; i < (1 << F); i += stride) {
        const float M = 1.0f + (float)i * (1.0f / (float)(1 << F));
        const float qe = __fdiv_rn(M, c.qs), q0 = __fmul_rn(M, p);
        const int e = (int)((__float_as_uint(qe) >> 23) & 0xffu) - 127;
#pragma unroll
        for (int k = 0; k < 7; ++k) {
            const int j = kBinades[k] - e;
            const uint32_t two = __nv_cvt_float2_to_fp8x2(make_float2(scale_pow2(qe, j), scale_pow2(q0, j)),
                                                          __NV_SATFINITE, __NV_E4M3);
            ok &= ((two ^ (two >> 8)) & 0xffu) == 0u;
        }
    }
    return ok;
}

// The last scale the search ran for on this device, per storage type, with
// its outcome: the scale's bits in the high half, the multiplier's bits in
// the low half (0: the product does not apply).  Written and read as one
// 64-bit word, so a reader sees one search's outcome whole; a write by a
// CTA of the current grid is seen by later grids (kernel boundaries order
// it) and maybe by CTAs of this one, which is harmless either way: the
// outcome for a scale is the same whoever computes it.  (Internal linkage:
// each translation unit that includes this keeps its own.)
static __device__ unsigned long long g_plain_memo[2];
template <DT T> __device__ __forceinline__ unsigned long long plain_memo_load() {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(&g_plain_memo[T == DT::BF16 ? 0 : 1]) : "memory");
    return v;
}
template <DT T> __device__ __forceinline__ void plain_memo_store(unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(&g_plain_memo[T == DT::BF16 ? 0 : 1]), "l"(v) : "memory");
}
__device__ __forceinline__ bool plain_memo_hit(unsigned long long m, const QuantE4M3 &c) {
    return c.fast && (uint32_t)(m >> 32) == __float_as_uint(c.qs);
}

// The CTA's search for a plain-product multiplier: candidates r, r -+ 1 ulp,
// r -+ 2 ulp in turn, each checked by all threads and closed by a barrier
// (every thread of the CTA calls it, for an ordinary positive scale).
// Returns the multiplier's bits, 0 if every candidate fails.  Out of line:
// it runs only when the memo misses, and kept apart it leaves the kernel's
// main path as it is.
template <DT T>
__device__ __noinline__ uint32_t quant_plain_search(float qs, float qr, int first, int stride) {
    QuantE4M3 c{};
    c.qs = qs;
    c.qr = qr;
    c.fast = true;
    for (int t = 0; t < kPlainTries; ++t) {
        const float p = plain_candidate(qr, t);
        if (__syncthreads_and(quant_plain_share<T>(c, p, first, stride))) return __float_as_uint(p);
    }
    return 0u;
}

// The CTA's decision between the plain product and the other forms (every
// thread of the CTA calls it, after a barrier that published memo_s: thread
// 0's plain_memo_load()).  A memo hit takes the recorded outcome; a miss
// searches and thread 0 records the outcome.  Sets c.plain and c.rp.
template <DT T>
__device__ __forceinline__ void quant_pick_plain(QuantE4M3 &c, const unsigned long long *memo_s, int first,
                                                 int stride) {
    const unsigned long long m = *memo_s;
    uint32_t rp = 0u;
    if (plain_memo_hit(m, c)) {
        rp = (uint32_t)m;
    } else if (c.fast) {
        rp = quant_plain_search<T>(c.qs, c.qr, first, stride);
        if (first == 0) plain_memo_store<T>(((unsigned long long)__float_as_uint(c.qs) << 32) | rp);
    }
    c.plain = rp != 0u;
    c.rp = c.plain ? __uint_as_float(rp) : c.qr;
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

// the e4m3 codes of 4 storage values (2 packed pairs), in memory order, when
// the product alone gives them (c.plain)
template <DT T>
__device__ __forceinline__ uint32_t quant4_e4m3_plain(const uint32_t *o, const QuantE4M3 &c) {
    const f2_t r2 = f2(c.rp, c.rp);
    const f2_t p01 = f2_mul(f2(lo_f32<T>(o[0]), hi_f32<T>(o[0])), r2);
    const f2_t p23 = f2_mul(f2(lo_f32<T>(o[1]), hi_f32<T>(o[1])), r2);
    float q0, q1, q2, q3;
    f2_split(p01, q0, q1);
    f2_split(p23, q2, q3);
    const uint32_t q01 = __nv_cvt_float2_to_fp8x2(make_float2(q0, q1), __NV_SATFINITE, __NV_E4M3);
    const uint32_t q23 = __nv_cvt_float2_to_fp8x2(make_float2(q2, q3), __NV_SATFINITE, __NV_E4M3);
    return (q01 & 0xffffu) | (q23 << 16);
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
    return c.plain ? quant4_e4m3_plain<T>(o, c) : c.fast ? quant4_e4m3_fast<T>(o, c) : quant4_e4m3_window<T>(o, c);
}

}  // namespace adaln
