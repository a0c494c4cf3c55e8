// Contiguous-rows kernel of the norm + modulate chains (one warp per row);
// instantiated per storage type, norm and gate in ln_rows_*.cu (eight
// translation units that compile in parallel).  Every global access of a row is 8 bytes (one
// logical lane's vec4 chunk), so rows only need 8-byte aligned starts.
#pragma once
#include "ln_common.cuh"
#include "quant_e4m3.cuh"

#include <type_traits>

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
// RMS: RMSNorm instead of LayerNorm.  Each lane sums x*x over its chunks
// (square and sum rounded separately), the same butterfly folds the sums
// with plain additions, rstd = rsqrt_rn(ss / D + eps), and the output pass
// is the LayerNorm's with mean 0 (x - 0 is x exactly).  Masked tail lanes
// hold zeros, which add nothing.
//
// OPSH: the modulate operands op = round(1 + scale) and shift of all B
// samples are computed once per CTA into shared memory (B * D * 4 bytes, at
// most kOpshMaxBytes), interleaved per column pair as (op, shift), so the
// output pass reads one 16-byte shared word per lane chunk instead of two
// global loads and an add per column pair.  Otherwise scale and shift are
// read from global memory (L2) in the output pass, at
// b * s_scale_b + n * s_scale_n (per-token rows, e.g. the chunks of a
// [B, S, 6D] modulation table, have s_scale_n != 0 and never use the table).
constexpr int kOpshMaxBytes = 32 * 1024;

// GM (gate mode): with a gate (GM != GATE_NONE) the row is first
// r = round(x + round(gate * y)) (the residual gate-add chain, x and y
// contiguous), written to r_out, and the norm and modulate run on r: one
// read of x and y, one write of r and out.  The gate of (b, n) sits at
// b * s_gate_b + n * s_gate_n: a row (GATE_ROW) or one value (GATE_SCALAR,
// a per-token [B, S, 1] gate).  GATE_ROW with OPSH: the rows are one per
// sample and join the shared table after the op / shift pairs (B * D * 2
// more bytes; the whole table stays within kOpshMaxBytes).
enum GateMode : int { GATE_NONE = 0, GATE_ROW = 1, GATE_SCALAR = 2 };

// E4M3: the output is static FP8, e4m3(y / *qscale) of each storage value
// y of the chain (binary32 division, round to nearest even, saturating at
// +-448): one byte per element, 4 per lane chunk.
struct RowsParams {
    uint16_t *out;
    const uint16_t *x;
    int64_t rows, B, N;
    int D;
    int64_t sxB, sxN;
    const uint16_t *scale;
    int64_t s_scale_b, s_scale_n;
    const uint16_t *shift;
    int64_t s_shift_b, s_shift_n;
    float eps;
    const uint16_t *y;
    const uint16_t *gate;
    int64_t s_gate_b, s_gate_n;
    uint16_t *r_out;
    const float *qscale;
};

// NI <= 8 (D <= 4096): two CTAs per SM (at most 128 registers a thread);
// NI 9..12 (D <= 6144): one CTA per SM, the longer row in registers.
template <DT T, int NI, bool TAIL, bool OPSH, int GM, bool RMS, bool E4M3 = false>
__global__ void __launch_bounds__(kRowsThreads, NI <= 8 ? 2 : 1)
ln_rows_kernel(const RowsParams p) {
    constexpr bool GATE = GM != GATE_NONE;
    constexpr bool GTAB = OPSH && GM == GATE_ROW;      // gate rows in the shared table
    extern __shared__ __align__(16) uint32_t opsh[];  // OPSH: [b][column pair][op, shift] (+ GTAB: [b][pair] gate)
    // this CTA's rows, from launch parameters only: computed before waiting
    // on the previous kernel and passed through shared memory so that the
    // parameter reads (a constant-cache miss) stay ahead of the wait
    __shared__ int64_t cta_rows[2];
    if (threadIdx.x == 0) {
        const int64_t per = p.rows / gridDim.x, extra = p.rows % gridDim.x;
        cta_rows[0] = blockIdx.x * per + imin64(blockIdx.x, extra);
        cta_rows[1] = cta_rows[0] + per + (blockIdx.x < extra ? 1 : 0);
    }
    __syncthreads();
    // Without a gate and with one scale / shift row per sample, each warp asks
    // L2 for its first row of x before waiting on the previous kernel.  A
    // prefetch is a hint with no effect on what later loads return (L2 is
    // where every SM's global accesses meet), so the loads after the wait
    // still see that kernel's writes; the DRAM latency of the first rows
    // overlaps its tail instead.  (Measured: 2.7 % faster at (1, 4096, 4096)
    // and 3.8 % for the e4m3 output; with a gate or per-token rows the same
    // prefetches made the kernel slower, so those forms do without.)
    if constexpr (GM == GATE_NONE && OPSH) {
        if ((threadIdx.x & 31) == 0) {
            const int64_t row0 = cta_rows[0] + (threadIdx.x >> 5);
            if (row0 < cta_rows[1]) {
                const int64_t b0 = row0 / p.N, n0 = row0 - b0 * p.N;
                prefetch_l2(p.x + b0 * p.sxB + n0 * p.sxN, (uint64_t)p.D * 2);
            }
        }
        // and the scale / shift rows the shared table is built from
        if (threadIdx.x < 2 * p.B && threadIdx.x < 64) {
            const int64_t bb = threadIdx.x >> 1;
            prefetch_l2((threadIdx.x & 1) ? p.shift + bb * p.s_shift_b : p.scale + bb * p.s_scale_b,
                        (uint64_t)p.D * 2);
        }
    }
    // Everything below up to the wait depends on launch parameters only; the
    // first row's loads are the first thing after it (a 64-bit division or a
    // parameter read there delays every row of the call).
    const int u = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int D = p.D;
    const int64_t N = p.N;
    const int nvec = D >> 2;
    const float Df = (float)D;
    const int l0 = (u & 7) + 32 * (u >> 3);
    const int c0 = 4 * l0;  // element offset of lane l0 at step 0

    FoldPlan plan;
    if constexpr (!RMS) {
        if constexpr (TAIL) {
            plan = fold_plan_runtime(u, nvec);
        } else {
            plan = fold_plan_uniform(NI);
        }
    }
    bool vlast[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) vlast[s] = !TAIL || (128 * (NI - 1) + l0 + 8 * s < nvec);

    // rows are split evenly into contiguous ranges per CTA; warps of the CTA
    // take them round-robin
    const int64_t r0 = cta_rows[0], r1 = cta_rows[1];

    // xv[i][s] = the 4 elements of lane l0 + 8s at step i (2 registers)
    uint32_t xv[NI][4][2];
    auto row_x = [&](int64_t b, int64_t n) { return p.x + b * p.sxB + n * p.sxN + c0; };
    auto load_row = [&](const uint16_t *xr) {
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
    // (b, n) of the warp's row, advanced with the row (a division only when
    // the warp's next row lies in a later sample)
    int64_t row = r0 + warp;
    int64_t rb = row / N, rn = row - rb * N;
    auto next_bn = [&](int64_t &b, int64_t &n) {
        n += kRowsThreads / 32;
        if (n >= N) {
            const int64_t q = n / N;
            b += q;
            n -= q * N;
        }
    };
    const uint16_t *const x_first = row_x(rb, rn);
    pdl_wait();
    pdl_trigger();
    if (row < r1) load_row(x_first);
    // E4M3: the static scale (written by earlier work on the stream) and the
    // device's memo of the plain-product search, read once the first row is
    // on its way; the constants are computed while the table's loads are in
    // flight, the form is picked after the barrier that ends the table
    float qs_in = 0.0f;
    unsigned long long memo = 0;
    __shared__ unsigned long long memo_s;
    if constexpr (E4M3) {
        qs_in = *p.qscale;
        memo = plain_memo_load<T>();
    }
    QuantE4M3 qc{};
    auto quant_prepare = [&] {
        if constexpr (E4M3) {
            qc = quant_setup<T>(qs_in);
            if (threadIdx.x == 0) memo_s = memo;
        }
    };
    if constexpr (E4M3 && !OPSH) {
        quant_prepare();
        __syncthreads();
        quant_pick_plain<T>(qc, &memo_s, threadIdx.x, kRowsThreads);
    }

    if constexpr (OPSH) {
        // all loads of a batch in flight before any is used
        constexpr int kFill = 8;
        const int half = D / 2, npairs = (int)p.B * half;  // npairs <= kOpshMaxBytes / 8
        for (int base = 0; base < npairs; base += kFill * kRowsThreads) {
            uint32_t s2[kFill], h2[kFill], g2[kFill];
#pragma unroll
            for (int k = 0; k < kFill; ++k) {
                const int e = base + k * kRowsThreads + threadIdx.x;
                if (e < npairs) {
                    const int bb = p.B == 1 ? 0 : e / half, cp = e - bb * half;
                    asm("ld.global.nc.b32 %0, [%1];" : "=r"(s2[k]) : "l"(p.scale + bb * p.s_scale_b + 2 * cp));
                    asm("ld.global.nc.b32 %0, [%1];" : "=r"(h2[k]) : "l"(p.shift + bb * p.s_shift_b + 2 * cp));
                    if constexpr (GTAB)
                        asm("ld.global.nc.b32 %0, [%1];" : "=r"(g2[k]) : "l"(p.gate + bb * p.s_gate_b + 2 * cp));
                }
            }
            if (base == 0) quant_prepare();
#pragma unroll
            for (int k = 0; k < kFill; ++k) {
                const int e = base + k * kRowsThreads + threadIdx.x;
                if (e < npairs) {
                    opsh[2 * e] = add16x2<T>(s2[k], one16x2<T>());
                    opsh[2 * e + 1] = h2[k];
                    if constexpr (GTAB) opsh[2 * npairs + e] = g2[k];
                }
            }
        }
        __syncthreads();
        if constexpr (E4M3) quant_pick_plain<T>(qc, &memo_s, threadIdx.x, kRowsThreads);
    }

    // the row loop, one copy per e4m3 quantiser form (chosen once per CTA;
    // a choice per row or per chunk inside one loop is slower)
    auto row_loop = [&](auto qform) {
        for (; row < r1; row += kRowsThreads / 32) {
            const int64_t b = rb, n = rn;
            int64_t bn = rb, nn = rn;  // the warp's next row
            next_bn(bn, nn);

            // pass 1: Welford (or the sum of squares) of lanes (s0, s1) and
            // (s2, s3), one f32x2 op each
            // (each instantiation uses some of these: the rest are marked maybe_unused)
            f2_t m01 = f2(0.f, 0.f), q01 = m01, q23 = m01;
            [[maybe_unused]] f2_t m23 = m01;
            [[maybe_unused]] const uint16_t *gr = nullptr;  // GATE: this row's gate row (or value)
            [[maybe_unused]] uint32_t gs = 0;               // GATE_SCALAR: the value in both halves
            if constexpr (GATE) gr = p.gate + b * p.s_gate_b + n * p.s_gate_n;
            if constexpr (GM == GATE_SCALAR) {
                const uint32_t g1 = ldg_u16(gr);
                gs = g1 | (g1 << 16);
            }
            static_for<0, NI>([&](auto I) {
                constexpr int i = decltype(I)::value;
                if constexpr (GATE) {
                    // this step's chunks become r = round(x + round(gate * y)), stored
                    const uint16_t *yr = p.y + row * (int64_t)D + c0;
                    uint16_t *rr_out = p.r_out + row * (int64_t)D + c0;
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        if (i < NI - 1 || vlast[s]) {
                            const int off = 512 * i + 32 * s;
                            uint32_t yv[2], gv[2];
                            ld_stream8(yv, yr + off);
                            if constexpr (GM == GATE_SCALAR) {
                                gv[0] = gv[1] = gs;
                            } else if constexpr (GTAB) {
                                const uint2 t = *reinterpret_cast<const uint2 *>(opsh + 2 * (int)(p.B * (D / 2)) + b * (D / 2) + (c0 + off) / 2);
                                gv[0] = t.x;
                                gv[1] = t.y;
                            } else {
                                ld_keep8(gv, gr + c0 + off);
                            }
                            xv[i][s][0] = add16x2<T>(xv[i][s][0], mul16x2<T>(gv[0], yv[0]));
                            xv[i][s][1] = add16x2<T>(xv[i][s][1], mul16x2<T>(gv[1], yv[1]));
                            st8(rr_out + off, xv[i][s]);
                        }
                    }
                }
                static_for<0, 4>([&](auto E) {
                    constexpr int e = decltype(E)::value;
                    [[maybe_unused]] constexpr float r = Rcp<4 * i + e + 1>::value;  // Welford 1/(count+1)
                    float a[4];
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        a[s] = (e & 1) ? hi_f32<T>(xv[i][s][e >> 1]) : lo_f32<T>(xv[i][s][e >> 1]);
                    if constexpr (RMS) {
                        // masked tail lanes hold zeros: adding 0 * 0 keeps the sum
                        const f2_t a01 = f2(a[0], a[1]), a23 = f2(a[2], a[3]);
                        q01 = f2_add(q01, f2_mul(a01, a01));
                        q23 = f2_add(q23, f2_mul(a23, a23));
                    } else if (!TAIL || i < NI - 1) {
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
            if (u == 0 && row + kRowsThreads / 32 < r1) prefetch_l2(p.x + bn * p.sxB + nn * p.sxN, (uint64_t)D * 2);

            float mean, m2;
            if constexpr (RMS) {
                mean = 0.0f;
                m2 = fold128_sum_s8(q01, q23);
            } else {
                fold128_s8(m01, q01, m23, q23, plan, mean, m2);
            }
            const float rstd = finish_rstd(m2, Df, p.eps);

            // pass 2: normalise, modulate, store
            [[maybe_unused]] const uint16_t *scr = p.scale + b * p.s_scale_b + n * p.s_scale_n + c0;
            [[maybe_unused]] const uint16_t *shr = p.shift + b * p.s_shift_b + n * p.s_shift_n + c0;
            // OPSH: (op, shift) of the column pairs from c0 on
            [[maybe_unused]] const uint32_t *ob = opsh + b * D + c0;
            [[maybe_unused]] uint16_t *orow = p.out + row * (int64_t)D + c0;
            [[maybe_unused]] uint8_t *orow8 = reinterpret_cast<uint8_t *>(p.out) + row * (int64_t)D + c0;  // E4M3
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
                        if constexpr (E4M3) {
                            constexpr int QF = decltype(qform)::value;
                            if constexpr (QF == 2) {
                                st4(orow8 + off, quant4_e4m3_plain<T>(o, qc));
                            } else if constexpr (QF == 1) {
                                st4(orow8 + off, quant4_e4m3_fast<T>(o, qc));
                            } else {
                                st4(orow8 + off, quant4_e4m3_window<T>(o, qc));
                            }
                        } else {
                            st8(orow + off, o);
                        }
                    }
                }
            }
            if (row + kRowsThreads / 32 < r1) load_row(row_x(bn, nn));
            rb = bn;
            rn = nn;
        }
    };
    if constexpr (E4M3) {
        if (qc.plain) {
            row_loop(std::integral_constant<int, 2>{});
        } else if (qc.fast) {
            row_loop(std::integral_constant<int, 1>{});
        } else {
            row_loop(std::integral_constant<int, 0>{});
        }
    } else {
        row_loop(std::integral_constant<int, 0>{});
    }
}

// the op / shift table of all samples (and with GATE_ROW the gate rows) in
// shared memory, in bytes
static inline int64_t rows_opsh_bytes(const LnArgs &a, int gm) { return a.B * a.D * (gm == GATE_ROW ? 6 : 4); }

// the op / shift rows (and with GATE_ROW the gate rows) are one per sample
// and the table fits in shared memory (the rows path already guarantees
// 8-byte aligned rows and even strides)
static inline bool rows_opsh_ok(const LnArgs &a, int gm) {
    const bool per_sample = a.N == 1 || (a.s_scale_n == 0 && a.s_shift_n == 0 && (gm != GATE_ROW || a.s_gate_n == 0));
    return per_sample && rows_opsh_bytes(a, gm) <= kOpshMaxBytes;
}

static inline int rows_gate_mode(const LnArgs &a) {
    return !a.gate ? GATE_NONE : (a.s_gate_d == 0 ? GATE_SCALAR : GATE_ROW);
}

template <DT T, int NI, bool TAIL, bool OPSH, int GM, bool RMS, bool E4M3>
static cudaError_t run_rows(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    auto k = ln_rows_kernel<T, NI, TAIL, OPSH, GM, RMS, E4M3>;
    // <= kOpshMaxBytes with OPSH (rows_opsh_ok), which leaves room for the
    // static shared memory under the 48 KiB a launch gets without opt-in
    const size_t smem = OPSH ? (size_t)rows_opsh_bytes(a, GM) : 0;
    const int64_t rows = a.B * a.N;
    const int64_t ctas_needed = (rows + kRowsThreads / 32 - 1) / (kRowsThreads / 32);
    const int64_t grid = imin64(ctas_needed, (int64_t)dev.sms * blocks_per_sm(k, kRowsThreads, smem));
    RowsParams p{(uint16_t *)a.out, (const uint16_t *)a.x, rows, a.B, a.N, (int)a.D, a.sxB, a.sxN,
                 (const uint16_t *)a.scale, a.s_scale_b, a.N == 1 ? 0 : a.s_scale_n,
                 (const uint16_t *)a.shift, a.s_shift_b, a.N == 1 ? 0 : a.s_shift_n, a.eps,
                 (const uint16_t *)a.y, (const uint16_t *)a.gate, a.s_gate_b, a.N == 1 ? 0 : a.s_gate_n,
                 (uint16_t *)a.r_out, a.qscale};
    return launch_k(k, dim3((unsigned)grid), dim3(kRowsThreads), smem, s, pdl, p);
}

template <DT T, int NI, int GM, bool RMS, bool E4M3>
static cudaError_t rows_tail(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    const bool tail = a.D % 512 != 0;
    if (rows_opsh_ok(a, GM))
        return tail ? run_rows<T, NI, true, true, GM, RMS, E4M3>(a, pdl, s, dev)
                    : run_rows<T, NI, false, true, GM, RMS, E4M3>(a, pdl, s, dev);
    return tail ? run_rows<T, NI, true, false, GM, RMS, E4M3>(a, pdl, s, dev)
                : run_rows<T, NI, false, false, GM, RMS, E4M3>(a, pdl, s, dev);
}

template <DT T, int GM, bool RMS, bool E4M3 = false>
static cudaError_t rows_vec(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    switch ((a.D + 511) / 512) {
        case 1: return rows_tail<T, 1, GM, RMS, E4M3>(a, pdl, s, dev);
        case 2: return rows_tail<T, 2, GM, RMS, E4M3>(a, pdl, s, dev);
        case 3: return rows_tail<T, 3, GM, RMS, E4M3>(a, pdl, s, dev);
        case 4: return rows_tail<T, 4, GM, RMS, E4M3>(a, pdl, s, dev);
        case 5: return rows_tail<T, 5, GM, RMS, E4M3>(a, pdl, s, dev);
        case 6: return rows_tail<T, 6, GM, RMS, E4M3>(a, pdl, s, dev);
        case 7: return rows_tail<T, 7, GM, RMS, E4M3>(a, pdl, s, dev);
        case 8: return rows_tail<T, 8, GM, RMS, E4M3>(a, pdl, s, dev);
        case 9: return rows_tail<T, 9, GM, RMS, E4M3>(a, pdl, s, dev);
        case 10: return rows_tail<T, 10, GM, RMS, E4M3>(a, pdl, s, dev);
        case 11: return rows_tail<T, 11, GM, RMS, E4M3>(a, pdl, s, dev);
        case 12: return rows_tail<T, 12, GM, RMS, E4M3>(a, pdl, s, dev);
    }
    return cudaErrorInvalidValue;
}

// the two gate forms of one (storage type, norm)
template <DT T, bool RMS>
static cudaError_t rows_gated(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    return rows_gate_mode(a) == GATE_SCALAR ? rows_vec<T, GATE_SCALAR, RMS>(a, pdl, s, dev)
                                            : rows_vec<T, GATE_ROW, RMS>(a, pdl, s, dev);
}

}  // namespace adaln
