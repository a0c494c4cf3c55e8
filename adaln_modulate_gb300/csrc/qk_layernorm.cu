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
// Mapping: one thread per (token, head) row.  The thread holds the row in
// registers (Dh/4 vec4 chunks = logical lanes), runs the 32 Welford chains,
// then the whole butterfly inside the thread on lane pairs (2k, 2k+1)
// packed in f32x2 registers:
//   offset 16: pairs k < 8 with k + 8,  offset 8: k < 4 with k + 4,
//   offset 4: k < 2 with k + 2,  offset 2: pair 0 with pair 1,
//   offset 1: the two halves of pair 0.
// Chan's coefficients depend only on Dh (lanes past Dh/4 hold nothing); for
// Dh = 128 they are 1/2 with the lower count 4, 8, 16, 32, 64.  The affine
// (w, b) of q and of k are staged in shared memory as binary32.
//
// RMS: the per-head QK RMSNorm of the same page (qk_rmsnorm_native): each
// lane sums x*x (square and sum rounded separately), the same butterfly
// folds the sums with plain additions, rstd = rsqrt_rn(ss / Dh + eps),
// u = rstd * x and out = round(w * u) (binary32 product, one storage
// rounding); there is no bias.
#include "common.cuh"
#include "kernels.h"
#include "ln_common.cuh"

namespace adaln {

constexpr int kQkThreads = 128;

// Butterfly of the 32-lane DAG inside one thread.  Before the stage of
// offset o, lane l (l < o) holds the lanes l + 2o t (t < 16/o) and its
// partner l + o the lanes l + o + 2o t; lanes at or past nl hold nothing.
__host__ __device__ constexpr float qk_count(int first, int o, int nl) {
    float n = 0.0f;
    for (int t = 0; t < 16 / o; ++t) n += (first + 2 * o * t < nl) ? 4.0f : 0.0f;
    return n;
}
__host__ __device__ constexpr float qk_coef(int l, int o, int nl) {
    const float a = qk_count(l, o, nl), b = qk_count(l + o, o, nl);
    return (a + b == 0.0f) ? 0.0f : b / (a + b);
}

// NL: logical lanes holding data (Dh / 4) as a compile-time constant (all
// fold coefficients are then constants), or 0 for a run-time Dh.
template <DT T, int NL, bool RMS>
__global__ void __launch_bounds__(kQkThreads)
qk_ln_kernel(uint16_t *q_out, const uint16_t *q, int64_t rows_q, uint16_t *k_out,
             const uint16_t *k, int64_t rows_k, int Dh, const uint16_t *wq, const uint16_t *bq,
             const uint16_t *wk, const uint16_t *bk, float eps) {
    __shared__ __align__(16) float aff[2][2][128];  // [q / k][w / b][column]
    const int nl = NL ? NL : (Dh >> 2);
    const float Df = (float)Dh;
    const int64_t total = rows_q + rows_k;
    const int64_t r_first = (int64_t)blockIdx.x * kQkThreads + threadIdx.x;

    uint32_t v[32][2];  // lane l: elements 4l..4l+3
    auto load_row = [&](int64_t r) {
        const uint16_t *src = r < rows_q ? q + r * Dh : k + (r - rows_q) * Dh;
#pragma unroll
        for (int l = 0; l < 32; ++l) {
            if (l < nl) {
                ld_stream8(v[l], src + 4 * l);
            } else {
                v[l][0] = v[l][1] = 0u;
            }
        }
    };
    // the thread's first row goes out first after the wait; the affine
    // parameters (needed only for the output) follow
    pdl_wait();
    pdl_trigger();
    if (r_first < total) load_row(r_first);
    for (int c = threadIdx.x; c < 128; c += kQkThreads) {
        const bool in = c < Dh;
        aff[0][0][c] = (in && rows_q) ? h_f32<T>(wq[c]) : 0.0f;
        aff[0][1][c] = (!RMS && in && rows_q) ? h_f32<T>(bq[c]) : 0.0f;
        aff[1][0][c] = (in && rows_k) ? h_f32<T>(wk[c]) : 0.0f;
        aff[1][1][c] = (!RMS && in && rows_k) ? h_f32<T>(bk[c]) : 0.0f;
    }
    __syncthreads();

    for (int64_t r = r_first; r < total; r += (int64_t)gridDim.x * kQkThreads) {
        const bool isq = r < rows_q;
        uint16_t *dst = isq ? q_out + r * Dh : k_out + (r - rows_q) * Dh;
        const float *w = aff[isq ? 0 : 1][0];
        const float *bb = aff[isq ? 0 : 1][1];
        if (r != r_first) load_row(r);

        // Welford of every lane (counts 1..4) on lane pairs (2k, 2k+1);
        // lanes at or past nl keep (0, 0).  RMS: the sums of squares in qq
        f2_t m[16], qq[16];
#pragma unroll
        for (int kp = 0; kp < 16; ++kp) {
            m[kp] = qq[kp] = f2(0.f, 0.f);
            if (RMS && 2 * kp < nl) {
                // the odd lane of a pair past the end holds zeros: it adds nothing
                const uint32_t *a0 = v[2 * kp], *a1 = v[2 * kp + 1];
                const f2_t e0 = f2(lo_f32<T>(a0[0]), lo_f32<T>(a1[0])), e1 = f2(hi_f32<T>(a0[0]), hi_f32<T>(a1[0]));
                const f2_t e2 = f2(lo_f32<T>(a0[1]), lo_f32<T>(a1[1])), e3 = f2(hi_f32<T>(a0[1]), hi_f32<T>(a1[1]));
                qq[kp] = f2_add(f2_add(f2_add(f2_mul(e0, e0), f2_mul(e1, e1)), f2_mul(e2, e2)), f2_mul(e3, e3));
            } else if (!RMS && 2 * kp < nl) {
                const uint32_t *a0 = v[2 * kp], *a1 = v[2 * kp + 1];
                push2(m[kp], qq[kp], f2(lo_f32<T>(a0[0]), lo_f32<T>(a1[0])), Rcp<1>::value);
                push2(m[kp], qq[kp], f2(hi_f32<T>(a0[0]), hi_f32<T>(a1[0])), Rcp<2>::value);
                push2(m[kp], qq[kp], f2(lo_f32<T>(a0[1]), lo_f32<T>(a1[1])), Rcp<3>::value);
                push2(m[kp], qq[kp], f2(hi_f32<T>(a0[1]), hi_f32<T>(a1[1])), Rcp<4>::value);
                if (2 * kp + 1 >= nl) {  // the odd lane of the pair is past the end
                    float x0, x1, y0, y1;
                    f2_split(m[kp], x0, x1);
                    f2_split(qq[kp], y0, y1);
                    m[kp] = f2(x0, 0.f);
                    qq[kp] = f2(y0, 0.f);
                }
            }
        }

        float mean, m2;
        if constexpr (RMS) {
            // offsets 16, 8, 4, 2 on lane pairs, offset 1 on the two halves
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1)
#pragma unroll
                for (int kp = 0; kp < o; ++kp) qq[kp] = f2_add(qq[kp], qq[kp + o]);
            float a0, a1;
            f2_split(qq[0], a0, a1);
            mean = 0.0f;
            m2 = __fadd_rn(a0, a1);
        } else if constexpr (NL != 0) {
            // offsets 16, 8, 4, 2 on lane pairs, offset 1 on the two halves
#define QK_STAGE(O)                                                                  \
    _Pragma("unroll") for (int kp = 0; kp < (O) / 2; ++kp) {                         \
        chan_p2(m[kp], qq[kp], m[kp + (O) / 2], qq[kp + (O) / 2],                   \
                f2(qk_coef(2 * kp, O, NL), qk_coef(2 * kp + 1, O, NL)),             \
                f2(qk_count(2 * kp, O, NL), qk_count(2 * kp + 1, O, NL)));          \
    }
            QK_STAGE(16)
            QK_STAGE(8)
            QK_STAGE(4)
            QK_STAGE(2)
#undef QK_STAGE
            float a0, a1, b0, b1;
            f2_split(m[0], a0, a1);
            f2_split(qq[0], b0, b1);
            chan_p(a0, b0, a1, b1, qk_coef(0, 1, NL), qk_count(0, 1, NL));
            mean = a0;
            m2 = b0;
        } else {
            float lm[32], lq[32];
#pragma unroll
            for (int kp = 0; kp < 16; ++kp) {
                f2_split(m[kp], lm[2 * kp], lm[2 * kp + 1]);
                f2_split(qq[kp], lq[2 * kp], lq[2 * kp + 1]);
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
#pragma unroll
                for (int l = 0; l < o; ++l) {
                    const float a = qk_count(l, o, nl), b = qk_count(l + o, o, nl);
                    const float n = __fadd_rn(a, b);
                    const float c = (n == 0.0f) ? 0.0f : __fdiv_rn(b, n);
                    chan_p(lm[l], lq[l], lm[l + o], lq[l + o], c, a);
                }
            }
            mean = lm[0];
            m2 = lq[0];
        }
        const float rstd = rsqrt_rn(__fadd_rn(__fdiv_rn(m2, Df), eps));

        // out = round(fma(w, rstd * (x - mean), b)); RMS: round(w * (rstd * x))
        const f2_t mm = f2(mean, mean), rr = f2(rstd, rstd);
        uint32_t o[32][2];
#pragma unroll
        for (int l = 0; l < 32; ++l) {
            if (l < nl) {
                const float4 w4 = *reinterpret_cast<const float4 *>(w + 4 * l);
                const float4 b4 = *reinterpret_cast<const float4 *>(bb + 4 * l);
                float x0, x1, x2, x3, y0, y1, y2, y3;
                unpack_again<T>(v[l][0], x0, x1);
                unpack_again<T>(v[l][1], x2, x3);
                f2_t u01 = f2_mul(f2_sub(f2(x0, x1), mm), rr);
                f2_t u23 = f2_mul(f2_sub(f2(x2, x3), mm), rr);
                if constexpr (RMS) {
                    u01 = f2_mul(f2(w4.x, w4.y), u01);
                    u23 = f2_mul(f2(w4.z, w4.w), u23);
                } else {
                    u01 = f2_fma(f2(w4.x, w4.y), u01, f2(b4.x, b4.y));
                    u23 = f2_fma(f2(w4.z, w4.w), u23, f2(b4.z, b4.w));
                }
                f2_split(u01, y0, y1);
                f2_split(u23, y2, y3);
                o[l][0] = pack_rn<T>(y0, y1);
                o[l][1] = pack_rn<T>(y2, y3);
            }
        }
#pragma unroll
        for (int l = 0; l < 32; ++l)
            if (l < nl) st8(dst + 4 * l, o[l]);
    }
}

// ---------------------------------------------------------------------
// Dh = 128, two threads per row.  Thread t (= 0, 1) of a row holds the lane
// pairs (4k + 2t, 4k + 2t + 1), k = 0..7: one 16-byte access per k, and the
// two threads of a row cover 32 contiguous bytes.  The butterfly: offsets
// 16, 8, 4 (k bits) inside the thread on f32x2 lane pairs (j = 0, 1),
// offset 2 (the thread bit) with one shuffle of the pair, offset 1 (j)
// inside the thread.  A warp takes 16 rows per iteration; the loop is
// uniform across the warp (threads past the end compute on zeros and store
// nothing), so every shuffle sees the full warp.
// ---------------------------------------------------------------------

template <DT T, bool RMS>
__global__ void __launch_bounds__(kQkThreads)
qk_ln_pair_kernel(uint16_t *q_out, const uint16_t *q, int64_t rows_q, uint16_t *k_out,
                  const uint16_t *k, int64_t rows_k, const uint16_t *wq, const uint16_t *bq,
                  const uint16_t *wk, const uint16_t *bk, float eps) {
    __shared__ __align__(16) float aff[2][2][128];  // [q / k][w / b][column]
    constexpr int NL = 32;
    // ask L2 for the warp's first 16 rows before waiting on the previous
    // kernel (a hint only: loads after the wait still see its writes)
    if ((threadIdx.x & 31) == 0) {
        const int64_t total = rows_q + rows_k;
        const int64_t nb = (((int64_t)blockIdx.x * kQkThreads + threadIdx.x) >> 5) * 16;
        const int64_t ne = imin64(nb + 16, total);
        if (nb < rows_q) prefetch_l2(q + nb * 128, (uint64_t)(imin64(ne, rows_q) - nb) * 256);
        const int64_t ks = nb > rows_q ? nb : rows_q;
        if (ne > ks) prefetch_l2(k + (ks - rows_q) * 128, (uint64_t)(ne - ks) * 256);
    }
    const int t = threadIdx.x & 1;
    const int64_t total = rows_q + rows_k;
    const int64_t w0 = (((int64_t)blockIdx.x * kQkThreads + threadIdx.x) >> 5) * 16;
    const int64_t wstride = ((int64_t)gridDim.x * kQkThreads >> 5) * 16;
    const int rin = (threadIdx.x & 31) >> 1;  // row of this thread within the warp's 16

    uint32_t v[8][4];  // k: lanes 4k + 2t (v[k][0..1]) and 4k + 2t + 1 (v[k][2..3])
    auto load_rows = [&](int64_t r) {
        const uint16_t *src = r < rows_q ? q + r * 128 : k + (r - rows_q) * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            if (r < total) {
                asm volatile("ld.global.nc.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(v[kk][0]), "=r"(v[kk][1]), "=r"(v[kk][2]), "=r"(v[kk][3])
                             : "l"(src + 16 * kk + 8 * t));
            } else {
                v[kk][0] = v[kk][1] = v[kk][2] = v[kk][3] = 0u;
            }
        }
    };
    // the warp's first 16 rows go out first after the wait; the affine
    // parameters (needed only for the output) follow
    pdl_wait();
    pdl_trigger();
    load_rows(w0 + rin);
    for (int c = threadIdx.x; c < 128; c += kQkThreads) {
        aff[0][0][c] = rows_q ? h_f32<T>(wq[c]) : 0.0f;
        aff[0][1][c] = (!RMS && rows_q) ? h_f32<T>(bq[c]) : 0.0f;
        aff[1][0][c] = rows_k ? h_f32<T>(wk[c]) : 0.0f;
        aff[1][1][c] = (!RMS && rows_k) ? h_f32<T>(bk[c]) : 0.0f;
    }
    __syncthreads();

    for (int64_t rbase = w0; rbase < total; rbase += wstride) {
        const int64_t r = rbase + rin;
        const bool active = r < total;
        const bool isq = r < rows_q;
        uint16_t *dst = isq ? q_out + r * 128 : k_out + (r - rows_q) * 128;
        const float *w = aff[isq ? 0 : 1][0];
        const float *bb = aff[isq ? 0 : 1][1];
        if (rbase != w0) load_rows(r);

        // Welford of lane pair (4k + 2t, 4k + 2t + 1), one f32x2 chain per k
        // (RMS: the sums of squares in qq)
        f2_t m[8], qq[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t *a0 = v[kk], *a1 = v[kk] + 2;
            m[kk] = qq[kk] = f2(0.f, 0.f);
            if constexpr (RMS) {
                const f2_t e0 = f2(lo_f32<T>(a0[0]), lo_f32<T>(a1[0])), e1 = f2(hi_f32<T>(a0[0]), hi_f32<T>(a1[0]));
                const f2_t e2 = f2(lo_f32<T>(a0[1]), lo_f32<T>(a1[1])), e3 = f2(hi_f32<T>(a0[1]), hi_f32<T>(a1[1]));
                qq[kk] = f2_add(f2_add(f2_add(f2_mul(e0, e0), f2_mul(e1, e1)), f2_mul(e2, e2)), f2_mul(e3, e3));
                continue;
            }
            push2(m[kk], qq[kk], f2(lo_f32<T>(a0[0]), lo_f32<T>(a1[0])), Rcp<1>::value);
            push2(m[kk], qq[kk], f2(hi_f32<T>(a0[0]), hi_f32<T>(a1[0])), Rcp<2>::value);
            push2(m[kk], qq[kk], f2(lo_f32<T>(a0[1]), lo_f32<T>(a1[1])), Rcp<3>::value);
            push2(m[kk], qq[kk], f2(hi_f32<T>(a0[1]), hi_f32<T>(a1[1])), Rcp<4>::value);
        }
        // these rows have arrived: ask L2 for the warp's next 16 rows now, so
        // that their DRAM reads overlap this iteration's fold and stores
        if ((threadIdx.x & 31) == 0 && rbase + wstride < total) {
            const int64_t nb = rbase + wstride, ne = imin64(nb + 16, total);
            if (nb < rows_q) prefetch_l2(q + nb * 128, (uint64_t)(imin64(ne, rows_q) - nb) * 256);
            const int64_t ks = nb > rows_q ? nb : rows_q;
            if (ne > ks) prefetch_l2(k + (ks - rows_q) * 128, (uint64_t)(ne - ks) * 256);
        }
        float mean, rstd;
        if constexpr (RMS) {
            // offsets 16, 8, 4 inside the thread, 2 across the thread pair, 1 on the halves
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) qq[kk] = f2_add(qq[kk], qq[kk + 4]);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) qq[kk] = f2_add(qq[kk], qq[kk + 2]);
            qq[0] = f2_add(qq[0], qq[1]);
            qq[0] = f2_add(qq[0], __shfl_xor_sync(0xffffffffu, qq[0], 1));
            float a0, a1;
            f2_split(qq[0], a0, a1);
            mean = 0.0f;
            rstd = rsqrt_rn(__fadd_rn(__fdiv_rn(__fadd_rn(a0, a1), 128.0f), eps));
        } else {
            // offsets 16, 8, 4: k with k + 4, k + 2, k + 1 (all lane counts equal)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                chan_p2(m[kk], qq[kk], m[kk + 4], qq[kk + 4], f2(qk_coef(0, 16, NL), qk_coef(0, 16, NL)),
                        f2(qk_count(0, 16, NL), qk_count(0, 16, NL)));
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
                chan_p2(m[kk], qq[kk], m[kk + 2], qq[kk + 2], f2(qk_coef(0, 8, NL), qk_coef(0, 8, NL)),
                        f2(qk_count(0, 8, NL), qk_count(0, 8, NL)));
            chan_p2(m[0], qq[0], m[1], qq[1], f2(qk_coef(0, 4, NL), qk_coef(0, 4, NL)),
                    f2(qk_count(0, 4, NL), qk_count(0, 4, NL)));
            {  // offset 2: the partner thread holds lanes with the other t
                const f2_t pm = __shfl_xor_sync(0xffffffffu, m[0], 1);
                const f2_t pq = __shfl_xor_sync(0xffffffffu, qq[0], 1);
                const f2_t lo = t ? pm : m[0], up = t ? m[0] : pm;
                const f2_t delta = f2_sub(up, lo);
                const f2_t c2 = f2(qk_coef(0, 2, NL), qk_coef(0, 2, NL));
                m[0] = f2_fma(delta, c2, lo);
                qq[0] = f2_fma(f2_mul(f2_mul(delta, delta), f2(qk_count(0, 2, NL), qk_count(0, 2, NL))), c2,
                               f2_add(qq[0], pq));
            }
            float a0, a1, b0, b1;
            f2_split(m[0], a0, a1);
            f2_split(qq[0], b0, b1);
            chan_p(a0, b0, a1, b1, qk_coef(0, 1, NL), qk_count(0, 1, NL));  // offset 1
            mean = a0;
            rstd = rsqrt_rn(__fadd_rn(__fdiv_rn(b0, 128.0f), eps));
        }

        const f2_t mm = f2(mean, mean), rr = f2(rstd, rstd);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t o[4];
            const int col = 16 * kk + 8 * t;
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // lane 4k + 2t + h: columns col + 4h .. +3
                const float4 w4 = *reinterpret_cast<const float4 *>(w + col + 4 * h);
                const float4 b4 = *reinterpret_cast<const float4 *>(bb + col + 4 * h);
                float x0, x1, x2, x3, y0, y1, y2, y3;
                unpack_again<T>(v[kk][2 * h], x0, x1);
                unpack_again<T>(v[kk][2 * h + 1], x2, x3);
                f2_t u01 = f2_mul(f2_sub(f2(x0, x1), mm), rr);
                f2_t u23 = f2_mul(f2_sub(f2(x2, x3), mm), rr);
                if constexpr (RMS) {
                    u01 = f2_mul(f2(w4.x, w4.y), u01);
                    u23 = f2_mul(f2(w4.z, w4.w), u23);
                } else {
                    u01 = f2_fma(f2(w4.x, w4.y), u01, f2(b4.x, b4.y));
                    u23 = f2_fma(f2(w4.z, w4.w), u23, f2(b4.z, b4.w));
                }
                f2_split(u01, y0, y1);
                f2_split(u23, y2, y3);
                o[2 * h] = pack_rn<T>(y0, y1);
                o[2 * h + 1] = pack_rn<T>(y2, y3);
            }
            if (active) st16(dst + col, o);
        }
    }
}

template <DT T, bool RMS>
static cudaError_t run_qk_pair(const QkArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    auto kern = qk_ln_pair_kernel<T, RMS>;
    const int64_t total = a.rows_q + a.rows_k;
    const int64_t ctas = (total * 2 + kQkThreads - 1) / kQkThreads;
    const int64_t grid = imin64(ctas, (int64_t)dev.sms * blocks_per_sm(kern, kQkThreads, 0));
    return launch_k(kern, dim3((unsigned)grid), dim3(kQkThreads), 0, s, pdl, (uint16_t *)a.q_out,
                    (const uint16_t *)a.q, a.rows_q, (uint16_t *)a.k_out, (const uint16_t *)a.k,
                    a.rows_k, (const uint16_t *)a.wq, (const uint16_t *)a.bq, (const uint16_t *)a.wk,
                    (const uint16_t *)a.bk, a.eps);
}

template <DT T, int NL, bool RMS>
static cudaError_t run_qk(const QkArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    auto kern = qk_ln_kernel<T, NL, RMS>;
    const int64_t total = a.rows_q + a.rows_k;
    const int64_t ctas = (total + kQkThreads - 1) / kQkThreads;
    const int64_t grid = imin64(ctas, (int64_t)dev.sms * blocks_per_sm(kern, kQkThreads, 0));
    return launch_k(kern, dim3((unsigned)grid), dim3(kQkThreads), 0, s, pdl, (uint16_t *)a.q_out,
                    (const uint16_t *)a.q, a.rows_q, (uint16_t *)a.k_out, (const uint16_t *)a.k,
                    a.rows_k, (int)a.Dh, (const uint16_t *)a.wq, (const uint16_t *)a.bq,
                    (const uint16_t *)a.wk, (const uint16_t *)a.bk, a.eps);
}

static bool al(const void *p, int a) { return p == nullptr || ((uintptr_t)p % (uintptr_t)a) == 0; }

template <DT T, bool RMS>
static cudaError_t qk_dispatch(const QkArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    const bool a16 = al(a.q, 16) && al(a.k, 16) && al(a.q_out, 16) && al(a.k_out, 16);
    if (a.Dh == 128) return a16 ? run_qk_pair<T, RMS>(a, pdl, s, dev) : run_qk<T, 32, RMS>(a, pdl, s, dev);
    if (a.Dh == 64) return run_qk<T, 16, RMS>(a, pdl, s, dev);
    return run_qk<T, 0, RMS>(a, pdl, s, dev);
}

// LayerNorm with affine, or (a.rms) RMSNorm with a weight
cudaError_t launch_qk_head_layernorm(const QkArgs &a, int dtype, bool pdl, cudaStream_t s,
                                     const DeviceInfo &dev) {
    if (a.rms) return dtype == 0 ? qk_dispatch<DT::BF16, true>(a, pdl, s, dev) : qk_dispatch<DT::FP16, true>(a, pdl, s, dev);
    return dtype == 0 ? qk_dispatch<DT::BF16, false>(a, pdl, s, dev) : qk_dispatch<DT::FP16, false>(a, pdl, s, dev);
}

}  // namespace adaln
