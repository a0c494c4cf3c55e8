// Contiguous-rows kernel of ln_modulate (one warp per row); instantiated per
// storage type in ln_rows_bf16.cu / ln_rows_fp16.cu.
#pragma once
#include "ln_common.cuh"

namespace adaln {

// ---------------------------------------------------------------------
// contiguous rows: one warp per row
// ---------------------------------------------------------------------

constexpr int kRowsThreads = 256;

template <DT T, int VEC, int NI>
__global__ void __launch_bounds__(kRowsThreads)
ln_rows_kernel(uint16_t *out, const uint16_t *x, int64_t rows, int64_t N, int D, int64_t sxB,
               int64_t sxN, const uint16_t *scale, int64_t s_scale_b, const uint16_t *shift,
               int64_t s_shift_b, float eps) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nvec = D >> 2;
    const float Df = (float)D;

    // sub-lane s of this thread is logical lane 4*lane + s; in the last step
    // its chunk 128*(NI-1) + 4*lane + s exists only below D/4
    bool vlast[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) vlast[s] = 128 * (NI - 1) + 4 * lane + s < nvec;
    const bool full_last = vlast[3];
    float cnt[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) cnt[s] = 4.0f * (float)(NI - 1) + (vlast[s] ? 4.0f : 0.0f);

    // rows are split evenly into contiguous ranges per CTA; warps of the CTA
    // take them round-robin
    const int64_t per = rows / gridDim.x, extra = rows % gridDim.x;
    const int64_t r0 = blockIdx.x * per + imin64(blockIdx.x, extra);
    const int64_t r1 = r0 + per + (blockIdx.x < extra ? 1 : 0);

    for (int64_t row = r0 + warp; row < r1; row += kRowsThreads / 32) {
        const int64_t b = row / N;
        const int64_t n = row - b * N;
        const uint16_t *xr = x + b * sxB + n * sxN;

        uint32_t xv[NI][8];
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const uint16_t *p = xr + 512 * i + 16 * lane;
            if (i < NI - 1 || full_last) {
                ld16el_stream<VEC>(xv[i], p);
            } else {
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    if (vlast[s]) {
                        ld_stream8(&xv[i][2 * s], p + 4 * s);
                    } else {
                        xv[i][2 * s] = 0u;
                        xv[i][2 * s + 1] = 0u;
                    }
                }
            }
        }

        // pass 1: serial Welford per logical lane, two lanes per f32x2 op
        f2_t m01 = f2(0.f, 0.f), q01 = m01, m23 = m01, q23 = m01;
        static_for<0, NI>([&](auto I) {
            constexpr int i = decltype(I)::value;
            static_for<0, 4>([&](auto E) {
                constexpr int e = decltype(E)::value;
                constexpr float r = Rcp<4 * i + e + 1>::value;
                const uint32_t *v = xv[i];
                float a0, a1, a2, a3;
                if constexpr ((e & 1) == 0) {
                    a0 = lo_f32<T>(v[e >> 1]);
                    a1 = lo_f32<T>(v[2 + (e >> 1)]);
                    a2 = lo_f32<T>(v[4 + (e >> 1)]);
                    a3 = lo_f32<T>(v[6 + (e >> 1)]);
                } else {
                    a0 = hi_f32<T>(v[e >> 1]);
                    a1 = hi_f32<T>(v[2 + (e >> 1)]);
                    a2 = hi_f32<T>(v[4 + (e >> 1)]);
                    a3 = hi_f32<T>(v[6 + (e >> 1)]);
                }
                if (i < NI - 1 || full_last) {
                    push2(m01, q01, f2(a0, a1), r);
                    push2(m23, q23, f2(a2, a3), r);
                } else {
                    f2_t nm01 = m01, nq01 = q01, nm23 = m23, nq23 = q23;
                    push2(nm01, nq01, f2(a0, a1), r);
                    push2(nm23, nq23, f2(a2, a3), r);
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

        // fold: logical offsets 16, 8, 4 = lane xor 4, 2, 1; offsets 2, 1
        // inside the thread; offsets 64, 32 = lane xor 16, 8
        Stat st[4];
        f2_split(m01, st[0].mean, st[1].mean);
        f2_split(m23, st[2].mean, st[3].mean);
        f2_split(q01, st[0].m2, st[1].m2);
        f2_split(q23, st[2].m2, st[3].m2);
#pragma unroll
        for (int s = 0; s < 4; ++s) st[s].cnt = cnt[s];
        const Stat f = fold128_k4(st);
        const float mean = f.mean;
        const float rstd = finish_rstd(f.m2, Df, eps);

        // pass 2: normalise, modulate, store
        const uint16_t *scr = scale + b * s_scale_b;
        const uint16_t *shr = shift + b * s_shift_b;
        uint16_t *orow = out + row * (int64_t)D;
        const f2_t mm = f2(mean, mean), rr = f2(rstd, rstd);
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const int col = 512 * i + 16 * lane;
            const bool full = (i < NI - 1 || full_last);
            uint32_t sc[8], sh[8], o[8];
            if (full) {
                ld16el_keep<VEC>(sc, scr + col);
                ld16el_keep<VEC>(sh, shr + col);
            } else {
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    if (vlast[s]) {
                        ld_keep8(&sc[2 * s], scr + col + 4 * s);
                        ld_keep8(&sh[2 * s], shr + col + 4 * s);
                    } else {
                        sc[2 * s] = sc[2 * s + 1] = 0u;
                        sh[2 * s] = sh[2 * s + 1] = 0u;
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                float xl, xh;
                unpack_again<T>(xv[i][k], xl, xh);
                f2_t v = f2_mul(f2_sub(f2(xl, xh), mm), rr);
                float y0, y1;
                f2_split(v, y0, y1);
                const uint32_t y = pack_rn<T>(y0, y1);
                const uint32_t op = add16x2<T>(sc[k], one16x2<T>());
                o[k] = add16x2<T>(mul16x2<T>(y, op), sh[k]);
            }
            if (full) {
                st16el<VEC>(orow + col, o);
            } else {
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    if (vlast[s]) st8(orow + col + 4 * s, &o[2 * s]);
            }
        }
    }
    pdl_trigger();
}

template <DT T, int VEC, int NI>
static cudaError_t run_rows(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    auto k = ln_rows_kernel<T, VEC, NI>;
    const int64_t rows = a.B * a.N;
    const int64_t ctas_needed = (rows + kRowsThreads / 32 - 1) / (kRowsThreads / 32);
    const int64_t grid = imin64(ctas_needed, (int64_t)dev.sms * blocks_per_sm(k, kRowsThreads, 0));
    return launch_k(k, dim3((unsigned)grid), dim3(kRowsThreads), 0, s, pdl, (uint16_t *)a.out,
                    (const uint16_t *)a.x, rows, a.N, (int)a.D, a.sxB, a.sxN,
                    (const uint16_t *)a.scale, a.s_scale_b, (const uint16_t *)a.shift, a.s_shift_b,
                    a.eps);
}

template <DT T, int VEC>
static cudaError_t rows_ni(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    switch ((a.D + 511) / 512) {
        case 1: return run_rows<T, VEC, 1>(a, pdl, s, dev);
        case 2: return run_rows<T, VEC, 2>(a, pdl, s, dev);
        case 3: return run_rows<T, VEC, 3>(a, pdl, s, dev);
        case 4: return run_rows<T, VEC, 4>(a, pdl, s, dev);
        case 5: return run_rows<T, VEC, 5>(a, pdl, s, dev);
        case 6: return run_rows<T, VEC, 6>(a, pdl, s, dev);
        case 7: return run_rows<T, VEC, 7>(a, pdl, s, dev);
        case 8: return run_rows<T, VEC, 8>(a, pdl, s, dev);
    }
    return cudaErrorInvalidValue;
}

template <DT T>
static cudaError_t rows_vec(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    switch (ln_rows_vec_bytes(a)) {
        case 32: return rows_ni<T, 32>(a, pdl, s, dev);
        case 16: return rows_ni<T, 16>(a, pdl, s, dev);
        case 8: return rows_ni<T, 8>(a, pdl, s, dev);
    }
    return cudaErrorInvalidValue;
}

}  // namespace adaln
