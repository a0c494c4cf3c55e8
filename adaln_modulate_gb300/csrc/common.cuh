// Device helpers shared by the sm_103a kernels of the fused DiT chains.
//
// Every floating-point step of the fixed rounding DAG is written with an
// explicit round-to-nearest operation (intrinsic or PTX), so nvcc never
// contracts a multiply and an add into an FMA or reassociates anything.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace adaln {

enum class DT : int { BF16 = 0, FP16 = 1 };

__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

// ---------------------------------------------------------------- PDL

// With ADALN_FLAG_PDL the kernel is launched with programmatic stream
// serialisation; it must not read inputs before the preceding grid has
// completed.  Without the launch attribute both instructions are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel on the stream (launched with the attribute) start its
// CTAs as SMs free up; its own pdl_wait still waits for this whole grid to
// complete, so every kernel here triggers right after its pdl_wait.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ----------------------------------------------- 16-bit storage <-> f32

// Element 0 of a packed pair sits in the low 16 bits.
template <DT T> __device__ __forceinline__ float lo_f32(uint32_t p);
template <DT T> __device__ __forceinline__ float hi_f32(uint32_t p);
template <> __device__ __forceinline__ float lo_f32<DT::BF16>(uint32_t p) { return __uint_as_float(p << 16); }
template <> __device__ __forceinline__ float hi_f32<DT::BF16>(uint32_t p) { return __uint_as_float(p & 0xffff0000u); }
template <> __device__ __forceinline__ float lo_f32<DT::FP16>(uint32_t p) {
    return __half2float(__ushort_as_half((unsigned short)(p & 0xffffu)));
}
template <> __device__ __forceinline__ float hi_f32<DT::FP16>(uint32_t p) {
    return __half2float(__ushort_as_half((unsigned short)(p >> 16)));
}
template <DT T> __device__ __forceinline__ float h_f32(uint16_t h) { return lo_f32<T>((uint32_t)h); }

// The same conversions through different instructions.  A kernel that
// converts the same packed registers twice (statistics pass, then output
// pass) uses these in the second pass, so that the compiler recomputes the
// values instead of keeping every converted float alive in registers.
template <DT T> __device__ __forceinline__ void unpack_again(uint32_t p, float &lo, float &hi);
template <> __device__ __forceinline__ void unpack_again<DT::BF16>(uint32_t p, float &lo, float &hi) {
    uint32_t a, b;
    asm("prmt.b32 %0, %1, 0, 0x1044;" : "=r"(a) : "r"(p));
    asm("prmt.b32 %0, %1, 0, 0x3244;" : "=r"(b) : "r"(p));
    lo = __uint_as_float(a);
    hi = __uint_as_float(b);
}
template <> __device__ __forceinline__ void unpack_again<DT::FP16>(uint32_t p, float &lo, float &hi) {
    uint32_t a, b;
    asm("prmt.b32 %0, %1, 0, 0x4410;" : "=r"(a) : "r"(p));
    asm("prmt.b32 %0, %1, 0, 0x4432;" : "=r"(b) : "r"(p));
    asm("{ .reg .b16 h; cvt.u16.u32 h, %1; cvt.f32.f16 %0, h; }" : "=f"(lo) : "r"(a));
    asm("{ .reg .b16 h; cvt.u16.u32 h, %1; cvt.f32.f16 %0, h; }" : "=f"(hi) : "r"(b));
}

// round-to-nearest-even pack of two binary32 values: lo -> bits 0..15
template <DT T> __device__ __forceinline__ uint32_t pack_rn(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack_rn<DT::BF16>(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
template <> __device__ __forceinline__ uint32_t pack_rn<DT::FP16>(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
template <DT T> __device__ __forceinline__ uint16_t to16_rn(float v) {
    return (uint16_t)(pack_rn<T>(v, 0.0f) & 0xffffu);
}

// Packed 16-bit arithmetic, each lane rounded once to the storage type.
// For one add or one multiply of two storage values this equals binary32
// arithmetic followed by one storage rounding: binary32 carries at least
// 2p+2 significand bits for p = 8 (bf16) and p = 11 (fp16), so the double
// rounding is innocuous (Figueroa, "When is double rounding innocuous?",
// SIGNUM 1995).
template <DT T> __device__ __forceinline__ uint32_t add16x2(uint32_t a, uint32_t b);
template <DT T> __device__ __forceinline__ uint32_t mul16x2(uint32_t a, uint32_t b);
template <> __device__ __forceinline__ uint32_t add16x2<DT::BF16>(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
template <> __device__ __forceinline__ uint32_t mul16x2<DT::BF16>(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
template <> __device__ __forceinline__ uint32_t add16x2<DT::FP16>(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
template <> __device__ __forceinline__ uint32_t mul16x2<DT::FP16>(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// 1.0 in both lanes
template <DT T> __device__ __forceinline__ uint32_t one16x2() {
    return T == DT::BF16 ? 0x3f803f80u : 0x3c003c00u;
}

// ------------------------------------------------------ packed binary32

typedef unsigned long long f2_t;  // two binary32 lanes: x in bits 0..31

__device__ __forceinline__ f2_t f2(float x, float y) {
    f2_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ void f2_split(f2_t v, float &x, float &y) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(v));
}
__device__ __forceinline__ f2_t f2_sub(f2_t a, f2_t b) {
    f2_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2_t f2_mul(f2_t a, f2_t b) {
    f2_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2_t f2_fma(f2_t a, f2_t b, f2_t c) {
    f2_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// ------------------------------------------------ global memory access

// Streaming (read-once) loads of 8/16/32 bytes, not allocated in L1.
__device__ __forceinline__ void ld_stream8(uint32_t *r, const void *p) {
    asm volatile("ld.global.nc.L1::no_allocate.v2.b32 {%0, %1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1]) : "l"(p));
}
__device__ __forceinline__ void ld_stream16(uint32_t *r, const void *p) {
    asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "l"(p));
}
__device__ __forceinline__ void ld_stream32(uint32_t *r, const void *p) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]),
                   "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]) : "l"(p));
}
// Loads of small rows re-read by many warps (scale / shift / gate / bias /
// affine weights).  These rows are read-only for the whole kernel and the
// host has checked that no output overlaps them, so the asm is not
// volatile: the compiler may hoist, batch and overlap these loads.
__device__ __forceinline__ void ld_keep8(uint32_t *r, const void *p) {
    asm("ld.global.nc.v2.b32 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "l"(p));
}
// 4 bytes, not allocated in L1 (4 e4m3 outputs)
__device__ __forceinline__ void st4(void *p, uint32_t r) {
    asm volatile("st.global.L1::no_allocate.b32 [%0], %1;" ::"l"(p), "r"(r) : "memory");
}

// one 16-bit value (a per-token gate), zero-extended
__device__ __forceinline__ uint32_t ldg_u16(const uint16_t *p) {
    unsigned short v;
    asm("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ void ld_keep16(uint32_t *r, const void *p) {
    asm("ld.global.nc.v4.b32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "l"(p));
}
__device__ __forceinline__ void ld_keep32(uint32_t *r, const void *p) {
    asm("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]),
          "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]) : "l"(p));
}
// Output stores of 8/16/32 bytes, not allocated in L1 (no kernel here reads
// its output back).
__device__ __forceinline__ void st8(void *p, const uint32_t *r) {
    asm volatile("st.global.L1::no_allocate.v2.b32 [%0], {%1, %2};" :: "l"(p), "r"(r[0]), "r"(r[1]) : "memory");
}
__device__ __forceinline__ void st16(void *p, const uint32_t *r) {
    asm volatile("st.global.L1::no_allocate.v4.b32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]) : "memory");
}
__device__ __forceinline__ void st32(void *p, const uint32_t *r) {
    asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 :: "l"(p), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]),
                    "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]) : "memory");
}

// Asynchronous global -> shared copy of 16 bytes (Ampere-style cp.async,
// bypassing L1) of which only src_bytes (<= 16) are read and the rest is
// zero-filled; completed per thread with commit / wait groups.
__device__ __forceinline__ void cp_async16_zfill(void *smem, const void *gmem, int src_bytes) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Ask L2 to fetch the 16-byte aligned part of [p, p + bytes) ahead of the
// loads that will read it: one bulk request, no registers, nothing to wait
// for.
__device__ __forceinline__ void prefetch_l2(const void *p, uint64_t bytes) {
    const uint64_t a = (uint64_t)p, lo = (a + 15) & ~15ull, hi = (a + bytes) & ~15ull;
    if (hi > lo)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(lo), "r"((uint32_t)(hi - lo)) : "memory");
}

// ------------------------------------------- Welford / Chan statistics

// 1/n rounded to nearest binary32, as a compile-time constant: the
// division is evaluated by the compiler front end in IEEE binary32.
template <int N> struct Rcp {
    static constexpr float value = 1.0f / static_cast<float>(N);
};
template <int E> __device__ __forceinline__ constexpr float rcp_const() { return Rcp<E>::value; }

struct Stat {
    float mean, m2, cnt;
};

// Chan's pairwise combine of the lower lane's state a and the upper lane's
// state b: n = na + nb, coef = nb / n (0 when n == 0), delta = mb - ma,
// mean = fma(delta, coef, ma), m2 = fma(delta^2 * na, coef, m2a + m2b).
__device__ __forceinline__ Stat chan(const Stat &a, const Stat &b) {
    Stat o;
    float n = __fadd_rn(a.cnt, b.cnt);
    float coef = (n == 0.0f) ? 0.0f : __fdiv_rn(b.cnt, n);
    float delta = __fsub_rn(b.mean, a.mean);
    o.mean = __fmaf_rn(delta, coef, a.mean);
    float dda = __fmul_rn(__fmul_rn(delta, delta), a.cnt);
    o.m2 = __fmaf_rn(dda, coef, __fadd_rn(a.m2, b.m2));
    o.cnt = n;
    return o;
}
// Butterfly stage over a warp lane bit: both partners end with
// chan(lower, upper).
__device__ __forceinline__ Stat shfl_stage(const Stat &s, int xor_mask, unsigned mask = 0xffffffffu) {
    Stat p;
    p.mean = __shfl_xor_sync(mask, s.mean, xor_mask);
    p.m2 = __shfl_xor_sync(mask, s.m2, xor_mask);
    p.cnt = __shfl_xor_sync(mask, s.cnt, xor_mask);
    const bool lower = (threadIdx.x & xor_mask) == 0;
    return lower ? chan(s, p) : chan(p, s);
}

// ----------------------------------------------- 1/sqrt, rounded to nearest

// 1/sqrt(x) rounded to nearest binary32: CUDA's __frsqrt_rn, which the CUDA
// math API specifies in round-to-nearest-even mode, i.e. the correctly
// rounded result.  A GPU test checks it bit for bit against an exact
// evaluation on every binary32 in [1, 4) and on random inputs over a wide
// exponent range.
__device__ __forceinline__ float rsqrt_rn(float x) { return __frsqrt_rn(x); }

}  // namespace adaln
