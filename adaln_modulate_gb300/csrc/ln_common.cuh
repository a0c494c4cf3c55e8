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

// The 128-lane fold when a warp holds all lanes, 4 per thread (thread u has
// logical lanes 4u..4u+3 in st[0..3]): offsets 16, 8, 4 are thread xor 4, 2,
// 1; offsets 2, 1 are inside the thread; offsets 64, 32 are thread xor 16,
// 8.  Every thread returns the merged state of all 128 lanes.
__device__ __forceinline__ Stat fold128_k4(Stat *st) {
#pragma unroll
    for (int s = 0; s < 4; ++s) st[s] = shfl_stage(st[s], 4);
#pragma unroll
    for (int s = 0; s < 4; ++s) st[s] = shfl_stage(st[s], 2);
#pragma unroll
    for (int s = 0; s < 4; ++s) st[s] = shfl_stage(st[s], 1);
    Stat f = chan(chan(st[0], st[2]), chan(st[1], st[3]));
    f = shfl_stage(f, 16);
    return shfl_stage(f, 8);
}

// Welford count of logical lane l (of 128) after pass 1: 4 per chunk
__device__ __forceinline__ float lane_count128(int l, int nvec) {
    return l < nvec ? 4.0f * (float)((nvec - 1 - l) / 128 + 1) : 0.0f;
}

__device__ __forceinline__ float finish_rstd(float m2, float Df, float eps) {
    return rsqrt_cr(__fadd_rn(__fdiv_rn(m2, Df), eps));
}


static inline bool ln_aligned(const void *p, int a) { return ((uintptr_t)p % (uintptr_t)a) == 0; }
static inline bool ln_mult(int64_t v, int64_t a) { return v % a == 0; }

int ln_rows_vec_bytes(const LnArgs &a);
constexpr int kRowsMaxNI = 8;     // contiguous rows in registers: D <= 4096
constexpr int kTokensMaxNI = 12;  // tokens tile in shared memory: D <= 6144
cudaError_t ln_rows_bf16(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev);
cudaError_t ln_rows_fp16(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev);
cudaError_t ln_tokens_launch(const LnArgs &a, int dtype, bool pdl, cudaStream_t s, const DeviceInfo &dev);
cudaError_t ln_generic_launch(const LnArgs &a, int dtype, bool pdl, cudaStream_t s, const DeviceInfo &dev);

}  // namespace adaln
