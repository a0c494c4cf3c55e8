// Per-head q/k LayerNorm with affine for sm_103a, q and k in one launch.
//
// Follows the "qk_head_layernorm" entry of the SGLang Diffusion "Fused
// Kernels" page (Normalization table: per-head LayerNorm on q/k, bit-exact)
// and PR #34008 "实现拆解" 1 (GLM-Image attention: q and k normalised by one
// kernel).  Rounding DAG: 32 logical lanes, lane l holds elements 4l..4l+3,
// serial Welford per lane, butterfly 16, 8, 4, 2, 1 with Chan's combine,
// var = m2 / Dh, rstd = rsqrt_rn(var + eps), out = round(fma(w, u, b)) with
// u = rstd * (x - mean) in binary32.
//
// Mapping: 8 threads per row, 4 logical lanes (16 consecutive elements, one
// 32-byte access) per thread; a warp normalises 4 rows at a time.  Logical
// offsets 16, 8, 4 are thread xor 4, 2, 1 inside the 8-thread group and
// offsets 2, 1 are inside the thread.
#include "common.cuh"
#include "kernels.h"

namespace adaln {

constexpr int kQkThreads = 256;

__device__ __forceinline__ void qk_push2(f2_t &m, f2_t &q, f2_t v, float r) {
    f2_t d = f2_sub(v, m);
    f2_t m1 = f2_fma(d, f2(r, r), m);
    q = f2_fma(d, f2_sub(v, m1), q);
    m = m1;
}

template <DT T> __device__ __forceinline__ void qk_load_affine(float *wf, float *bf, const uint16_t *w,
                                                              const uint16_t *b, int col0, const bool *valid) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        uint32_t wr[2] = {0u, 0u}, br[2] = {0u, 0u};
        if (valid[s]) {
            ld_keep8(wr, w + col0 + 4 * s);
            ld_keep8(br, b + col0 + 4 * s);
        }
        wf[4 * s + 0] = lo_f32<T>(wr[0]);
        wf[4 * s + 1] = hi_f32<T>(wr[0]);
        wf[4 * s + 2] = lo_f32<T>(wr[1]);
        wf[4 * s + 3] = hi_f32<T>(wr[1]);
        bf[4 * s + 0] = lo_f32<T>(br[0]);
        bf[4 * s + 1] = hi_f32<T>(br[0]);
        bf[4 * s + 2] = lo_f32<T>(br[1]);
        bf[4 * s + 3] = hi_f32<T>(br[1]);
    }
}

// FULL: Dh == 128 with 32-byte aligned rows (one v8 access per thread)
template <DT T, bool FULL>
__global__ void __launch_bounds__(kQkThreads)
qk_ln_kernel(uint16_t *q_out, const uint16_t *q, int64_t rows_q, uint16_t *k_out,
             const uint16_t *k, int64_t rows_k, int Dh, const uint16_t *wq, const uint16_t *bq,
             const uint16_t *wk, const uint16_t *bk, float eps) {
    pdl_wait();
    const int sub = threadIdx.x & 7;
    const int col0 = 16 * sub;
    const int nvec = Dh >> 2;
    const float Df = (float)Dh;
    bool valid[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) valid[s] = FULL || (4 * sub + s < nvec);
    float cnt[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) cnt[s] = valid[s] ? 4.0f : 0.0f;

    const int64_t total = rows_q + rows_k;
    // the row loop is uniform across the warp (its 4 groups take 4
    // consecutive rows); groups past the end compute on zeros and store
    // nothing, so every shuffle sees the full warp
    const int64_t w0 = (((int64_t)blockIdx.x * kQkThreads + threadIdx.x) >> 5) * 4;
    const int64_t wstride = ((int64_t)gridDim.x * kQkThreads >> 5) * 4;
    const int grp = (threadIdx.x >> 3) & 3;

    // affine of the tensor currently being processed (rows of q come first)
    int cur = -1;
    float wf[16], bf[16];

    for (int64_t rb = w0; rb < total; rb += wstride) {
        const int64_t r = rb + grp;
        const bool active = r < total;
        const bool isq = r < rows_q;
        const int which = isq ? 0 : 1;
        if (active && which != cur) {
            qk_load_affine<T>(wf, bf, isq ? wq : wk, isq ? bq : bk, col0, valid);
            cur = which;
        }
        const uint16_t *src = isq ? q + r * Dh : k + (r - rows_q) * Dh;
        uint16_t *dst = isq ? q_out + r * Dh : k_out + (r - rows_q) * Dh;

        uint32_t v[8];
        if (!active) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) v[kk] = 0u;
        } else if (FULL) {
            ld_stream32(v, src + col0);
        } else {
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                if (valid[s]) {
                    ld_stream8(&v[2 * s], src + col0 + 4 * s);
                } else {
                    v[2 * s] = v[2 * s + 1] = 0u;
                }
            }
        }

        // Welford over the 4 elements of each logical lane (counts 1..4)
        f2_t m01 = f2(0.f, 0.f), q01 = m01, m23 = m01, q23 = m01;
        const float rc[4] = {Rcp<1>::value, Rcp<2>::value, Rcp<3>::value, Rcp<4>::value};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int h = e >> 1;
            float a0, a1, a2, a3;
            if ((e & 1) == 0) {
                a0 = lo_f32<T>(v[h]);
                a1 = lo_f32<T>(v[2 + h]);
                a2 = lo_f32<T>(v[4 + h]);
                a3 = lo_f32<T>(v[6 + h]);
            } else {
                a0 = hi_f32<T>(v[h]);
                a1 = hi_f32<T>(v[2 + h]);
                a2 = hi_f32<T>(v[4 + h]);
                a3 = hi_f32<T>(v[6 + h]);
            }
            qk_push2(m01, q01, f2(a0, a1), rc[e]);
            qk_push2(m23, q23, f2(a2, a3), rc[e]);
        }
        Stat st[4];
        f2_split(m01, st[0].mean, st[1].mean);
        f2_split(m23, st[2].mean, st[3].mean);
        f2_split(q01, st[0].m2, st[1].m2);
        f2_split(q23, st[2].m2, st[3].m2);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            if (!valid[s]) st[s].mean = st[s].m2 = 0.0f;  // a lane past Dh pushed nothing
            st[s].cnt = cnt[s];
        }
#pragma unroll
        for (int s = 0; s < 4; ++s) st[s] = shfl_stage(st[s], 4);
#pragma unroll
        for (int s = 0; s < 4; ++s) st[s] = shfl_stage(st[s], 2);
#pragma unroll
        for (int s = 0; s < 4; ++s) st[s] = shfl_stage(st[s], 1);
        const Stat f = chan(chan(st[0], st[2]), chan(st[1], st[3]));
        const float rstd = rsqrt_cr(__fadd_rn(__fdiv_rn(f.m2, Df), eps));

        const f2_t mm = f2(f.mean, f.mean), rr = f2(rstd, rstd);
        uint32_t o[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            f2_t u = f2(lo_f32<T>(v[kk]), hi_f32<T>(v[kk]));
            u = f2_mul(f2_sub(u, mm), rr);
            u = f2_fma(f2(wf[2 * kk], wf[2 * kk + 1]), u, f2(bf[2 * kk], bf[2 * kk + 1]));
            float y0, y1;
            f2_split(u, y0, y1);
            o[kk] = pack_rn<T>(y0, y1);
        }
        if (!active) {
            // nothing to store
        } else if (FULL) {
            st32(dst + col0, o);
        } else {
#pragma unroll
            for (int s = 0; s < 4; ++s)
                if (valid[s]) st8(dst + col0 + 4 * s, &o[2 * s]);
        }
    }
    pdl_trigger();
}

template <DT T, bool FULL>
static cudaError_t run_qk(const QkArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    auto kern = qk_ln_kernel<T, FULL>;
    const int64_t total = a.rows_q + a.rows_k;
    const int64_t ctas = (total * 8 + kQkThreads - 1) / kQkThreads;  // 32 rows per CTA pass
    const int64_t grid = imin64(ctas, (int64_t)dev.sms * blocks_per_sm(kern, kQkThreads, 0));
    return launch_k(kern, dim3((unsigned)grid), dim3(kQkThreads), 0, s, pdl, (uint16_t *)a.q_out,
                    (const uint16_t *)a.q, a.rows_q, (uint16_t *)a.k_out, (const uint16_t *)a.k,
                    a.rows_k, (int)a.Dh, (const uint16_t *)a.wq, (const uint16_t *)a.bq,
                    (const uint16_t *)a.wk, (const uint16_t *)a.bk, a.eps);
}

static bool al(const void *p, int a) { return p == nullptr || ((uintptr_t)p % (uintptr_t)a) == 0; }

cudaError_t launch_qk_head_layernorm(const QkArgs &a, int dtype, bool pdl, cudaStream_t s,
                                     const DeviceInfo &dev) {
    const bool full = a.Dh == 128 && al(a.q, 32) && al(a.k, 32) && al(a.q_out, 32) && al(a.k_out, 32);
    if (dtype == 0)
        return full ? run_qk<DT::BF16, true>(a, pdl, s, dev) : run_qk<DT::BF16, false>(a, pdl, s, dev);
    return full ? run_qk<DT::FP16, true>(a, pdl, s, dev) : run_qk<DT::FP16, false>(a, pdl, s, dev);
}

}  // namespace adaln
