// Contiguous-rows kernel of ln_modulate (one warp per row); instantiated per
// storage type in ln_rows_bf16.cu / ln_rows_fp16.cu.  Every access is 8
// bytes (one logical lane's vec4 chunk), so rows only need 8-byte aligned
// starts.
#pragma once
#include "ln_common.cuh"

namespace adaln {

// ---------------------------------------------------------------------
// contiguous rows: one warp per row
// ---------------------------------------------------------------------

constexpr int kRowsThreads = 256;

// One warp per row.  Thread u holds the logical lanes l0 + 8s (s = 0..3,
// l0 = (u & 7) + 32 (u >> 3)); at step i lane l owns elements
// 4(128 i + l) .. +3, i.e. one 8-byte access per lane and step.  A warp's
// access for a given s covers 4 runs of 64 contiguous bytes.  TAIL: D is
// not a multiple of 512 (the last step masks lanes past D/4 and the fold
// coefficients are computed per thread).
template <DT T, int NI, bool TAIL>
__global__ void __launch_bounds__(kRowsThreads)
ln_rows_kernel(uint16_t *out, const uint16_t *x, int64_t rows, int64_t N, int D, int64_t sxB,
               int64_t sxN, const uint16_t *scale, int64_t s_scale_b, const uint16_t *shift,
               int64_t s_shift_b, float eps) {
    pdl_wait();
    const int u = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nvec = D >> 2;
    const float Df = (float)D;
    const int l0 = (u & 7) + 32 * (u >> 3);
    const int c0 = 4 * l0;  // element offset of lane l0 at step 0

    FoldPlan plan;
    if constexpr (TAIL) {
        plan = fold_plan_runtime(u, nvec);
    } else {
        plan = fold_plan_uniform(NI);
    }
    bool vlast[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) vlast[s] = !TAIL || (128 * (NI - 1) + l0 + 8 * s < nvec);

    // rows are split evenly into contiguous ranges per CTA; warps of the CTA
    // take them round-robin
    const int64_t per = rows / gridDim.x, extra = rows % gridDim.x;
    const int64_t r0 = blockIdx.x * per + imin64(blockIdx.x, extra);
    const int64_t r1 = r0 + per + (blockIdx.x < extra ? 1 : 0);

    for (int64_t row = r0 + warp; row < r1; row += kRowsThreads / 32) {
        const int64_t b = row / N;
        const int64_t n = row - b * N;
        const uint16_t *xr = x + b * sxB + n * sxN + c0;

        // xv[i][s] = the 4 elements of lane l0 + 8s at step i (2 registers)
        uint32_t xv[NI][4][2];
#pragma unroll
        for (int i = 0; i < NI; ++i) {
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                if (i < NI - 1 || vlast[s]) {
                    ld_stream8(xv[i][s], xr + 512 * i + 32 * s);
                } else {
                    xv[i][s][0] = xv[i][s][1] = 0u;
                }
            }
        }

        // pass 1: Welford of lanes (s0, s1) and (s2, s3), one f32x2 op each
        f2_t m01 = f2(0.f, 0.f), q01 = m01, m23 = m01, q23 = m01;
        static_for<0, NI>([&](auto I) {
            constexpr int i = decltype(I)::value;
            static_for<0, 4>([&](auto E) {
                constexpr int e = decltype(E)::value;
                constexpr float r = Rcp<4 * i + e + 1>::value;
                float a[4];
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    a[s] = (e & 1) ? hi_f32<T>(xv[i][s][e >> 1]) : lo_f32<T>(xv[i][s][e >> 1]);
                if (!TAIL || i < NI - 1) {
                    push2(m01, q01, f2(a[0], a[1]), r);
                    push2(m23, q23, f2(a[2], a[3]), r);
                } else {
                    // last step with masked lanes: keep the old state there
                    f2_t nm01 = m01, nq01 = q01, nm23 = m23, nq23 = q23;
                    push2(nm01, nq01, f2(a[0], a[1]), r);
                    push2(nm23, nq23, f2(a[2], a[3]), r);
                    float o[4], w[4], oq[4], wq[4];
                    f2_split(m01, o[0], o[1]);
                    f2_split(m23, o[2], o[3]);
                    f2_split(nm01, w[0], w[1]);
                    f2_split(nm23, w[2], w[3]);
                    f2_split(q01, oq[0], oq[1]);
                    f2_split(q23, oq[2], oq[3]);
                    f2_split(nq01, wq[0], wq[1]);
                    f2_split(nq23, wq[2], wq[3]);
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        o[s] = vlast[s] ? w[s] : o[s];
                        oq[s] = vlast[s] ? wq[s] : oq[s];
                    }
                    m01 = f2(o[0], o[1]);
                    m23 = f2(o[2], o[3]);
                    q01 = f2(oq[0], oq[1]);
                    q23 = f2(oq[2], oq[3]);
                }
            });
        });

        float mean, m2;
        fold128_s8(m01, q01, m23, q23, plan, mean, m2);
        const float rstd = finish_rstd(m2, Df, eps);

        // pass 2: normalise, modulate, store
        const uint16_t *scr = scale + b * s_scale_b + c0;
        const uint16_t *shr = shift + b * s_shift_b + c0;
        uint16_t *orow = out + row * (int64_t)D + c0;
        const f2_t mm = f2(mean, mean), rr = f2(rstd, rstd);
#pragma unroll
        for (int i = 0; i < NI; ++i) {
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                if (i < NI - 1 || vlast[s]) {
                    const int off = 512 * i + 32 * s;
                    uint32_t sc[2], sh[2], o[2];
                    ld_keep8(sc, scr + off);
                    ld_keep8(sh, shr + off);
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        float xl, xh;
                        unpack_again<T>(xv[i][s][k], xl, xh);
                        float y0, y1;
                        f2_split(f2_mul(f2_sub(f2(xl, xh), mm), rr), y0, y1);
                        const uint32_t op = add16x2<T>(sc[k], one16x2<T>());
                        o[k] = add16x2<T>(mul16x2<T>(pack_rn<T>(y0, y1), op), sh[k]);
                    }
                    st8(orow + off, o);
                }
            }
        }
    }
    pdl_trigger();
}

template <DT T, int NI, bool TAIL>
static cudaError_t run_rows(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    auto k = ln_rows_kernel<T, NI, TAIL>;
    const int64_t rows = a.B * a.N;
    const int64_t ctas_needed = (rows + kRowsThreads / 32 - 1) / (kRowsThreads / 32);
    const int64_t grid = imin64(ctas_needed, (int64_t)dev.sms * blocks_per_sm(k, kRowsThreads, 0));
    return launch_k(k, dim3((unsigned)grid), dim3(kRowsThreads), 0, s, pdl, (uint16_t *)a.out,
                    (const uint16_t *)a.x, rows, a.N, (int)a.D, a.sxB, a.sxN,
                    (const uint16_t *)a.scale, a.s_scale_b, (const uint16_t *)a.shift, a.s_shift_b,
                    a.eps);
}

template <DT T, int NI>
static cudaError_t rows_tail(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    return (a.D % 512 == 0) ? run_rows<T, NI, false>(a, pdl, s, dev) : run_rows<T, NI, true>(a, pdl, s, dev);
}

template <DT T>
static cudaError_t rows_vec(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    switch ((a.D + 511) / 512) {
        case 1: return rows_tail<T, 1>(a, pdl, s, dev);
        case 2: return rows_tail<T, 2>(a, pdl, s, dev);
        case 3: return rows_tail<T, 3>(a, pdl, s, dev);
        case 4: return rows_tail<T, 4>(a, pdl, s, dev);
        case 5: return rows_tail<T, 5>(a, pdl, s, dev);
        case 6: return rows_tail<T, 6>(a, pdl, s, dev);
        case 7: return rows_tail<T, 7>(a, pdl, s, dev);
        case 8: return rows_tail<T, 8>(a, pdl, s, dev);
    }
    return cudaErrorInvalidValue;
}

}  // namespace adaln
