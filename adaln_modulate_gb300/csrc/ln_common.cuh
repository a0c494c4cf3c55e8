// LayerNorm helpers shared by the ln_modulate kernels (see ln_modulate.cu
// for the rounding DAG they implement).
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace adaln {

template <int V> struct IC { static constexpr int value = V; };
template <int B, int E, typename F> __device__ __forceinline__ void static_for(F &&f) {
    if constexpr (B < E) {
        f(IC<B>{});
        static_for<B + 1, E>(f);
    }
}

// one serial Welford step on two independent lanes: d = v - mean,
// mean' = fma(d, r, mean), m2' = fma(d, v - mean', m2), r = 1/(count+1)
__device__ __forceinline__ void push2(f2_t &m, f2_t &q, f2_t v, float r) {
    f2_t d = f2_sub(v, m);
    f2_t m1 = f2_fma(d, f2(r, r), m);
    q = f2_fma(d, f2_sub(v, m1), q);
    m = m1;
}

__device__ __forceinline__ void push1(Stat &s, float v) {
    float d = __fsub_rn(v, s.mean);
    float c1 = __fadd_rn(s.cnt, 1.0f);
    float r = __fdiv_rn(1.0f, c1);
    float m1 = __fmaf_rn(d, r, s.mean);
    s.m2 = __fmaf_rn(d, __fsub_rn(v, m1), s.m2);
    s.mean = m1;
    s.cnt = c1;
}

// ---------------------------------------------------------------------
// The fold with the "stride-8" lane mapping: thread u of a warp holds the
// logical lanes l0 + 8s, s = 0..3, with l0 = (u & 7) + 32 (u >> 3).  The
// butterfly offsets then map to
//   16, 8      inside the thread (s bit 1, then s bit 0),
//   4, 2, 1    thread xor 4, 2, 1,
//   64, 32     thread xor 16, 8,
// so after the two in-thread stages only one state crosses threads.
//
// Chan's coefficient of a stage, coef = n_upper / (n_lower + n_upper), and
// the lower side's count n_lower depend only on D (the lanes' counts), not
// on the data; FoldPlan holds them for one thread.  When every lane holds
// the same number of chunks (D % 512 == 0) they are compile-time constants:
// coef = 1/2 exactly and n_lower doubles from 4*NI at every stage.
// ---------------------------------------------------------------------

struct FoldPlan {
    float c16[2], n16[2];  // in-thread offset 16: pairs (s0, s2), (s1, s3)
    float c8, n8;          // in-thread offset 8
    float c[5], n[5];      // offsets 4, 2, 1, 64, 32
};
static_assert(sizeof(FoldPlan) == 16 * sizeof(float), "FoldPlan is 16 floats");

__host__ __device__ constexpr FoldPlan fold_plan_uniform(int NI) {
    FoldPlan p{};
    const float n1 = 4.0f * (float)NI;
    p.c16[0] = p.c16[1] = 0.5f;
    p.n16[0] = p.n16[1] = n1;
    p.c8 = 0.5f;
    p.n8 = 2.0f * n1;
    float n = 4.0f * n1;
    for (int k = 0; k < 5; ++k) {
        p.c[k] = 0.5f;
        p.n[k] = n;
        n *= 2.0f;
    }
    return p;
}

// Sum of the Welford counts of the lanes first, first + stride, ...
// (n lanes).  Lane l (< 128) holds 4*(NI-1) + 4*[l < r] values, with
// NI = ceil(nvec / 128) chunk steps and r = nvec - 128*(NI-1) lanes that
// own a chunk in the last step.
__device__ __forceinline__ float ap_count(int first, int stride, int n, int ni, int r) {
    int below = 0;
    if (first < r) {
        below = (r - 1 - first) / stride + 1;
        below = below < n ? below : n;
    }
    return 4.0f * (float)((ni - 1) * n + below);
}

__device__ __forceinline__ void plan_coef(float a, float b, float &c, float &n_lower) {
    const float n = __fadd_rn(a, b);
    c = (n == 0.0f) ? 0.0f : __fdiv_rn(b, n);
    n_lower = a;
}

// Plan for thread u of a warp, any D.  Along this butterfly every merged
// lane set is an arithmetic progression (or two): before offset 16 the
// single lanes; before 8 {l, l+16}; before 4 stride 8; before 2 stride 4;
// before 1 stride 2; before 64 the 32 lanes of a group; before 32 two
// groups.
__device__ __forceinline__ FoldPlan fold_plan_runtime(int u, int nvec) {
    FoldPlan p;
    const int ni = (nvec + 127) / 128;
    const int r = nvec - 128 * (ni - 1);
    const int l0 = (u & 7) + 32 * (u >> 3);
    plan_coef(ap_count(l0, 1, 1, ni, r), ap_count(l0 + 16, 1, 1, ni, r), p.c16[0], p.n16[0]);
    plan_coef(ap_count(l0 + 8, 1, 1, ni, r), ap_count(l0 + 24, 1, 1, ni, r), p.c16[1], p.n16[1]);
    plan_coef(ap_count(l0, 16, 2, ni, r), ap_count(l0 + 8, 16, 2, ni, r), p.c8, p.n8);
    plan_coef(ap_count(l0 & ~4, 8, 4, ni, r), ap_count(l0 | 4, 8, 4, ni, r), p.c[0], p.n[0]);
    plan_coef(ap_count(l0 & ~6, 4, 8, ni, r), ap_count((l0 & ~6) | 2, 4, 8, ni, r), p.c[1], p.n[1]);
    plan_coef(ap_count(l0 & ~7, 2, 16, ni, r), ap_count((l0 & ~7) | 1, 2, 16, ni, r), p.c[2], p.n[2]);
    plan_coef(ap_count(l0 & 32, 1, 32, ni, r), ap_count((l0 & 32) + 64, 1, 32, ni, r), p.c[3], p.n[3]);
    plan_coef(ap_count(0, 1, 32, ni, r) + ap_count(64, 1, 32, ni, r),
              ap_count(32, 1, 32, ni, r) + ap_count(96, 1, 32, ni, r), p.c[4], p.n[4]);
    return p;
}

// Chan's combine with a precomputed coefficient: (ma, qa) is the lower
// lane's state and becomes the merged state.
__device__ __forceinline__ void chan_p(float &ma, float &qa, float mb, float qb, float coef, float na) {
    const float delta = __fsub_rn(mb, ma);
    const float m = __fmaf_rn(delta, coef, ma);
    qa = __fmaf_rn(__fmul_rn(__fmul_rn(delta, delta), na), coef, __fadd_rn(qa, qb));
    ma = m;
}

__device__ __forceinline__ f2_t f2_add(f2_t a, f2_t b) {
    f2_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// the same on two lane pairs at once: lower (ma, qa), upper (mb, qb)
__device__ __forceinline__ void chan_p2(f2_t &ma, f2_t &qa, f2_t mb, f2_t qb, f2_t coef, f2_t na) {
    const f2_t delta = f2_sub(mb, ma);
    const f2_t m = f2_fma(delta, coef, ma);
    qa = f2_fma(f2_mul(f2_mul(delta, delta), na), coef, f2_add(qa, qb));
    ma = m;
}

// butterfly stage across threads: both partners end with
// combine(lower, upper); `mask` is the thread-index bit of the stage
__device__ __forceinline__ void shfl_stage_p(float &m, float &q, int mask, float coef, float na) {
    const float pm = __shfl_xor_sync(0xffffffffu, m, mask);
    const float pq = __shfl_xor_sync(0xffffffffu, q, mask);
    const bool lower = (threadIdx.x & mask) == 0;
    const float lo = lower ? m : pm, up = lower ? pm : m;
    const float delta = __fsub_rn(up, lo);
    m = __fmaf_rn(delta, coef, lo);
    q = __fmaf_rn(__fmul_rn(__fmul_rn(delta, delta), na), coef, __fadd_rn(q, pq));
}

// Fold of the 4 lane states of every thread of a warp (stride-8 mapping):
// m01 / q01 hold lanes s0, s1 and m23 / q23 lanes s2, s3.  Returns the
// 128-lane (mean, m2) in every thread.
__device__ __forceinline__ void fold128_s8(f2_t m01, f2_t q01, f2_t m23, f2_t q23, const FoldPlan &p,
                                           float &mean, float &m2) {
    chan_p2(m01, q01, m23, q23, f2(p.c16[0], p.c16[1]), f2(p.n16[0], p.n16[1]));  // offset 16
    float m0, m1, q0, q1;
    f2_split(m01, m0, m1);
    f2_split(q01, q0, q1);
    chan_p(m0, q0, m1, q1, p.c8, p.n8);                                          // offset 8
    shfl_stage_p(m0, q0, 4, p.c[0], p.n[0]);
    shfl_stage_p(m0, q0, 2, p.c[1], p.n[1]);
    shfl_stage_p(m0, q0, 1, p.c[2], p.n[2]);
    shfl_stage_p(m0, q0, 16, p.c[3], p.n[3]);
    shfl_stage_p(m0, q0, 8, p.c[4], p.n[4]);
    mean = m0;
    m2 = q0;
}

// The same fold for two tokens at once: each f32x2 holds one lane's state of
// tokens A (x) and B (y), so every step is the per-token step of fold128_s8
// on both tokens in one instruction (the same IEEE operations in the same
// order for each token, hence the same bits).  s0..s3 are the thread's lanes
// l0, l0 + 8, l0 + 16, l0 + 24.
__device__ __forceinline__ void shfl_stage_p2(f2_t &m, f2_t &q, int mask, float coef, float na) {
    const f2_t pm = __shfl_xor_sync(0xffffffffu, m, mask);
    const f2_t pq = __shfl_xor_sync(0xffffffffu, q, mask);
    const bool lower = (threadIdx.x & mask) == 0;
    const f2_t lo = lower ? m : pm, up = lower ? pm : m;
    const f2_t delta = f2_sub(up, lo);
    m = f2_fma(delta, f2(coef, coef), lo);
    q = f2_fma(f2_mul(f2_mul(delta, delta), f2(na, na)), f2(coef, coef), f2_add(q, pq));
}

__device__ __forceinline__ void fold128_s8_x2(f2_t m0, f2_t q0, f2_t m1, f2_t q1, f2_t m2, f2_t q2, f2_t m3,
                                              f2_t q3, const FoldPlan &p, f2_t &mean, f2_t &m2out) {
    chan_p2(m0, q0, m2, q2, f2(p.c16[0], p.c16[0]), f2(p.n16[0], p.n16[0]));  // offset 16: (s0, s2)
    chan_p2(m1, q1, m3, q3, f2(p.c16[1], p.c16[1]), f2(p.n16[1], p.n16[1]));  //            (s1, s3)
    chan_p2(m0, q0, m1, q1, f2(p.c8, p.c8), f2(p.n8, p.n8));                  // offset 8
    shfl_stage_p2(m0, q0, 4, p.c[0], p.n[0]);
    shfl_stage_p2(m0, q0, 2, p.c[1], p.n[1]);
    shfl_stage_p2(m0, q0, 1, p.c[2], p.n[2]);
    shfl_stage_p2(m0, q0, 16, p.c[3], p.n[3]);
    shfl_stage_p2(m0, q0, 8, p.c[4], p.n[4]);
    mean = m0;
    m2out = q0;
}

// RMSNorm: the 128 lanes' sums of squares folded in the butterfly order of
// fold128_s8 (offsets 16 and 8 inside the thread, then 4, 2, 1, 64, 32
// across threads) with plain additions.  IEEE addition commutes, so both
// partners of a stage compute the same bits.  Returned in every thread.
__device__ __forceinline__ float fold128_sum_s8(f2_t s01, f2_t s23) {
    float a, b;
    f2_split(f2_add(s01, s23), a, b);  // offset 16: (s0 + s2, s1 + s3)
    float t = __fadd_rn(a, b);         // offset 8
    t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, 4));
    t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, 2));
    t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, 1));
    t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, 16));  // offset 64
    t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, 8));   // offset 32
    return t;
}

// rstd = rsqrt_rn(m2 / D + eps): var = m2 / D for the LayerNorm, and with
// m2 the sum of squares, ms = ss / D for the RMSNorm
__device__ __forceinline__ float finish_rstd(float m2, float Df, float eps) {
    return rsqrt_rn(__fadd_rn(__fdiv_rn(m2, Df), eps));
}


static inline bool ln_aligned(const void *p, int a) { return ((uintptr_t)p % (uintptr_t)a) == 0; }
static inline bool ln_mult(int64_t v, int64_t a) { return v % a == 0; }

bool ln_rows_ok(const LnArgs &a);
constexpr int kRowsMaxNI = 12;    // contiguous rows in registers: D <= 6144
constexpr int kTokensMaxNI = 12;  // tokens tile in shared memory: D <= 6144
// contiguous-rows kernels (ln_rows_*.cu): LayerNorm / RMSNorm, without or
// with the residual gate (a.gate; x, y, r_out, out contiguous)
#define ADALN_ROWS_DECL(name) cudaError_t name(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev);
ADALN_ROWS_DECL(rows_ln_bf16)
ADALN_ROWS_DECL(rows_ln_fp16)
ADALN_ROWS_DECL(rows_ln_gate_bf16)
ADALN_ROWS_DECL(rows_ln_gate_fp16)
ADALN_ROWS_DECL(rows_rms_bf16)
ADALN_ROWS_DECL(rows_rms_fp16)
ADALN_ROWS_DECL(rows_rms_gate_bf16)
ADALN_ROWS_DECL(rows_rms_gate_fp16)
ADALN_ROWS_DECL(rows_ln_fp8_bf16)  // LayerNorm, no gate, static FP8 output
ADALN_ROWS_DECL(rows_ln_fp8_fp16)
#undef ADALN_ROWS_DECL
cudaError_t ln_tokens_launch(const LnArgs &a, int dtype, bool pdl, cudaStream_t s, const DeviceInfo &dev);
cudaError_t ln_generic_launch(const LnArgs &a, int dtype, bool pdl, cudaStream_t s, const DeviceInfo &dev);

}  // namespace adaln
