// Contiguous-rows kernel of ln_modulate (one warp per row); instantiated per
// storage type in ln_rows_bf16.cu / ln_rows_fp16.cu.  Every global access is
// 8 bytes (one logical lane's vec4 chunk), so rows only need 8-byte aligned
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
//
// OPSH: the modulate operands op = round(1 + scale) and shift of all B
// samples are computed once per CTA into shared memory (B * D * 4 bytes, at
// most kOpshMaxBytes), interleaved per column pair as (op, shift), so the
// output pass reads one 16-byte shared word per lane chunk instead of two
// global loads and an add per column pair.  Otherwise scale and shift are
// read from global memory (L2) in the output pass.
constexpr int kOpshMaxBytes = 32 * 1024;

// GATE: the row is first r = round(x + round(gate * y)) (the residual
// gate-add chain, x and y contiguous), written to r_out, and the LayerNorm
// and modulate run on r: one read of x and y, one write of r and out.
// With OPSH the gate rows join the shared table (after the op / shift
// pairs, B * D * 2 more bytes; the whole table stays within kOpshMaxBytes).
struct RowsGate {
    const uint16_t *y;
    const uint16_t *gate;
    int64_t s_gate_b;
    uint16_t *r_out;
};

template <DT T, int NI, bool TAIL, bool OPSH, bool GATE>
__global__ void __launch_bounds__(kRowsThreads, 2)
ln_rows_kernel(uint16_t *out, const uint16_t *x, int64_t rows, int64_t B, int64_t N, int D,
               int64_t sxB, int64_t sxN, const uint16_t *scale, int64_t s_scale_b,
               const uint16_t *shift, int64_t s_shift_b, float eps, RowsGate g) {
    extern __shared__ __align__(16) uint32_t opsh[];  // OPSH: [b][column pair][op, shift] (+ GATE: [b][pair] gate)
    // this CTA's rows, from launch parameters only: computed before waiting
    // on the previous kernel and passed through shared memory so that the
    // parameter reads (a constant-cache miss) stay ahead of the wait
    __shared__ int64_t cta_rows[2];
    if (threadIdx.x == 0) {
        const int64_t per = rows / gridDim.x, extra = rows % gridDim.x;
        cta_rows[0] = blockIdx.x * per + imin64(blockIdx.x, extra);
        cta_rows[1] = cta_rows[0] + per + (blockIdx.x < extra ? 1 : 0);
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();
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
    const int64_t r0 = cta_rows[0], r1 = cta_rows[1];

    // xv[i][s] = the 4 elements of lane l0 + 8s at step i (2 registers)
    uint32_t xv[NI][4][2];
    auto load_row = [&](int64_t row) {
        const int64_t b = row / N;
        const uint16_t *xr = x + b * sxB + (row - b * N) * sxN + c0;
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
    };
    int64_t row = r0 + warp;
    if (row < r1) load_row(row);

    if constexpr (OPSH) {
        // all loads of a batch in flight before any is used
        constexpr int kFill = 8;
        const int half = D / 2, npairs = (int)B * half;  // npairs <= kOpshMaxBytes / 8
        for (int base = 0; base < npairs; base += kFill * kRowsThreads) {
            uint32_t s2[kFill], h2[kFill], g2[kFill];
#pragma unroll
            for (int k = 0; k < kFill; ++k) {
                const int e = base + k * kRowsThreads + threadIdx.x;
                if (e < npairs) {
                    const int bb = e / half, cp = e - bb * half;
                    asm("ld.global.nc.b32 %0, [%1];" : "=r"(s2[k]) : "l"(scale + bb * s_scale_b + 2 * cp));
                    asm("ld.global.nc.b32 %0, [%1];" : "=r"(h2[k]) : "l"(shift + bb * s_shift_b + 2 * cp));
                    if constexpr (GATE)
                        asm("ld.global.nc.b32 %0, [%1];" : "=r"(g2[k]) : "l"(g.gate + bb * g.s_gate_b + 2 * cp));
                }
            }
#pragma unroll
            for (int k = 0; k < kFill; ++k) {
                const int e = base + k * kRowsThreads + threadIdx.x;
                if (e < npairs) {
                    opsh[2 * e] = add16x2<T>(s2[k], one16x2<T>());
                    opsh[2 * e + 1] = h2[k];
                    if constexpr (GATE) opsh[2 * npairs + e] = g2[k];
                }
            }
        }
        __syncthreads();
    }

    for (; row < r1; row += kRowsThreads / 32) {
        const int64_t b = row / N;

        // pass 1: Welford of lanes (s0, s1) and (s2, s3), one f32x2 op each
        f2_t m01 = f2(0.f, 0.f), q01 = m01, m23 = m01, q23 = m01;
        static_for<0, NI>([&](auto I) {
            constexpr int i = decltype(I)::value;
            if constexpr (GATE) {
                // this step's chunks become r = round(x + round(gate * y)), stored
                const uint16_t *yr = g.y + row * (int64_t)D + c0;
                uint16_t *rr_out = g.r_out + row * (int64_t)D + c0;
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    if (i < NI - 1 || vlast[s]) {
                        const int off = 512 * i + 32 * s;
                        uint32_t yv[2], gv[2];
                        ld_stream8(yv, yr + off);
                        if constexpr (OPSH) {
                            const uint2 t = *reinterpret_cast<const uint2 *>(opsh + 2 * (int)(B * (D / 2)) + b * (D / 2) + (c0 + off) / 2);
                            gv[0] = t.x;
                            gv[1] = t.y;
                        } else {
                            ld_keep8(gv, g.gate + b * g.s_gate_b + c0 + off);
                        }
                        xv[i][s][0] = add16x2<T>(xv[i][s][0], mul16x2<T>(gv[0], yv[0]));
                        xv[i][s][1] = add16x2<T>(xv[i][s][1], mul16x2<T>(gv[1], yv[1]));
                        st8(rr_out + off, xv[i][s]);
                    }
                }
            }
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

        // this row has arrived: ask L2 for the warp's next row now, so that
        // its DRAM reads overlap this row's fold, output pass and stores
        if (u == 0 && row + kRowsThreads / 32 < r1) {
            const int64_t rn = row + kRowsThreads / 32, bn = rn / N;
            prefetch_l2(x + bn * sxB + (rn - bn * N) * sxN, (uint64_t)D * 2);
        }

        float mean, m2;
        fold128_s8(m01, q01, m23, q23, plan, mean, m2);
        const float rstd = finish_rstd(m2, Df, eps);

        // pass 2: normalise, modulate, store
        const uint16_t *scr = scale + b * s_scale_b + c0;
        const uint16_t *shr = shift + b * s_shift_b + c0;
        const uint32_t *ob = opsh + b * D + c0;  // OPSH: (op, shift) of the column pairs from c0 on
        uint16_t *orow = out + row * (int64_t)D + c0;
        const f2_t mm = f2(mean, mean), rr = f2(rstd, rstd);
#pragma unroll
        for (int i = 0; i < NI; ++i) {
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                if (i < NI - 1 || vlast[s]) {
                    const int off = 512 * i + 32 * s;
                    uint32_t op[2], sh[2], o[2];
                    if constexpr (OPSH) {
                        const uint4 t = *reinterpret_cast<const uint4 *>(ob + off);
                        op[0] = t.x;
                        sh[0] = t.y;
                        op[1] = t.z;
                        sh[1] = t.w;
                    } else {
                        uint32_t sc[2];
                        ld_keep8(sc, scr + off);
                        ld_keep8(sh, shr + off);
                        op[0] = add16x2<T>(sc[0], one16x2<T>());
                        op[1] = add16x2<T>(sc[1], one16x2<T>());
                    }
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        float xl, xh;
                        unpack_again<T>(xv[i][s][k], xl, xh);
                        float y0, y1;
                        f2_split(f2_mul(f2_sub(f2(xl, xh), mm), rr), y0, y1);
                        o[k] = add16x2<T>(mul16x2<T>(pack_rn<T>(y0, y1), op[k]), sh[k]);
                    }
                    st8(orow + off, o);
                }
            }
        }
        if (row + kRowsThreads / 32 < r1) load_row(row + kRowsThreads / 32);
    }
}

static inline int64_t rows_opsh_bytes(const LnArgs &a, bool gate) { return a.B * a.D * (gate ? 6 : 4); }

template <DT T, int NI, bool TAIL, bool OPSH, bool GATE>
static cudaError_t run_rows(const LnArgs &a, const RowsGate &g, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    auto k = ln_rows_kernel<T, NI, TAIL, OPSH, GATE>;
    // <= kOpshMaxBytes with OPSH (rows_opsh_ok), which leaves room for the
    // static shared memory under the 48 KiB a launch gets without opt-in
    const size_t smem = OPSH ? (size_t)rows_opsh_bytes(a, GATE) : 0;
    const int64_t rows = a.B * a.N;
    const int64_t ctas_needed = (rows + kRowsThreads / 32 - 1) / (kRowsThreads / 32);
    const int64_t grid = imin64(ctas_needed, (int64_t)dev.sms * blocks_per_sm(k, kRowsThreads, smem));
    return launch_k(k, dim3((unsigned)grid), dim3(kRowsThreads), smem, s, pdl, (uint16_t *)a.out,
                    (const uint16_t *)a.x, rows, a.B, a.N, (int)a.D, a.sxB, a.sxN,
                    (const uint16_t *)a.scale, a.s_scale_b, (const uint16_t *)a.shift, a.s_shift_b,
                    a.eps, g);
}

// the op / shift table of all samples (and with GATE the gate rows) fits in
// shared memory (the rows path already guarantees 8-byte aligned scale /
// shift and even strides)
static inline bool rows_opsh_ok(const LnArgs &a, bool gate) { return rows_opsh_bytes(a, gate) <= kOpshMaxBytes; }

template <DT T, int NI, bool GATE>
static cudaError_t rows_tail(const LnArgs &a, const RowsGate &g, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    const bool tail = a.D % 512 != 0;
    if (rows_opsh_ok(a, GATE))
        return tail ? run_rows<T, NI, true, true, GATE>(a, g, pdl, s, dev)
                    : run_rows<T, NI, false, true, GATE>(a, g, pdl, s, dev);
    return tail ? run_rows<T, NI, true, false, GATE>(a, g, pdl, s, dev)
                : run_rows<T, NI, false, false, GATE>(a, g, pdl, s, dev);
}

template <DT T, bool GATE>
static cudaError_t rows_vec(const LnArgs &a, const RowsGate &g, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    switch ((a.D + 511) / 512) {
        case 1: return rows_tail<T, 1, GATE>(a, g, pdl, s, dev);
        case 2: return rows_tail<T, 2, GATE>(a, g, pdl, s, dev);
        case 3: return rows_tail<T, 3, GATE>(a, g, pdl, s, dev);
        case 4: return rows_tail<T, 4, GATE>(a, g, pdl, s, dev);
        case 5: return rows_tail<T, 5, GATE>(a, g, pdl, s, dev);
        case 6: return rows_tail<T, 6, GATE>(a, g, pdl, s, dev);
        case 7: return rows_tail<T, 7, GATE>(a, g, pdl, s, dev);
        case 8: return rows_tail<T, 8, GATE>(a, g, pdl, s, dev);
    }
    return cudaErrorInvalidValue;
}

}  // namespace adaln
