// Norm + modulate for any strides and every option (LayerNorm or RMSNorm,
// per-sample or per-token operand rows, an optional residual gate in front):
// one CTA of 128 threads per row, thread l is logical lane l, scalar loads,
// plain binary32 code.  The path of last resort behind the rows and tokens
// kernels; same DAG, same bits.
#include <cuda_fp8.h>

#include "ln_common.cuh"

namespace adaln {

struct GenericParams {
    uint16_t *out;
    const uint16_t *x;
    int64_t B, N, D, sxB, sxN, sxD;
    const uint16_t *scale;
    int64_t s_scale_b, s_scale_n;
    const uint16_t *shift;
    int64_t s_shift_b, s_shift_n;
    float eps;
    const uint16_t *gate;  // null: no residual gate
    int64_t s_gate_b, s_gate_n, s_gate_d;
    const uint16_t *y;
    uint16_t *r_out;
    const float *qscale;  // set: out holds e4m3 bytes, e4m3(y / *qscale)
};

// Pass 1 reads x (and y, gate), forms v (r = round(x + round(gate * y)) with
// a gate, stored to r_out) and accumulates the lane's statistic over its
// chunks j = l, l + 128, ... in element order; pass 2 visits the same
// elements, re-reading x, or r_out as this thread stored it.  No thread
// reads an element another thread wrote, so r_out may alias x or y.
template <DT T, bool RMS>
__global__ void __launch_bounds__(128)
ln_generic_kernel(const GenericParams p) {
    __shared__ float xch[4][3];
    __shared__ float fin[2];
    const int l = threadIdx.x;
    const int64_t D = p.D, nvec = D >> 2;
    const float Df = (float)D;
    pdl_wait();
    pdl_trigger();
    const float qs = p.qscale ? *p.qscale : 1.0f;
    for (int64_t row = blockIdx.x; row < p.B * p.N; row += gridDim.x) {
        const int64_t b = row / p.N, n = row - b * p.N;
        const uint16_t *xr = p.x + b * p.sxB + n * p.sxN;
        const uint16_t *gr = p.gate ? p.gate + b * p.s_gate_b + n * p.s_gate_n : nullptr;
        const uint16_t *yr = p.gate ? p.y + row * D : nullptr;  // y and r_out only with a gate
        uint16_t *rr = p.gate ? p.r_out + row * D : nullptr;
        Stat s{0.f, 0.f, 0.f};
        float ss = 0.f;
        for (int64_t j = l; j < nvec; j += 128)
            for (int e = 0; e < 4; ++e) {
                const int64_t d = 4 * j + e;
                float v = h_f32<T>(xr[d * p.sxD]);
                if (gr) {
                    const float gy = h_f32<T>(to16_rn<T>(__fmul_rn(h_f32<T>(gr[d * p.s_gate_d]), h_f32<T>(yr[d]))));
                    const uint16_t r16 = to16_rn<T>(__fadd_rn(v, gy));
                    rr[d] = r16;
                    v = h_f32<T>(r16);
                }
                if constexpr (RMS) {
                    ss = __fadd_rn(ss, __fmul_rn(v, v));
                } else {
                    push1(s, v);
                }
            }
        if constexpr (RMS) {
            for (int off = 16; off >= 1; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
            if ((l & 31) == 0) xch[l >> 5][0] = ss;
        } else {
            for (int off = 16; off >= 1; off >>= 1) s = shfl_stage(s, off);
            if ((l & 31) == 0) {
                xch[l >> 5][0] = s.mean;
                xch[l >> 5][1] = s.m2;
                xch[l >> 5][2] = s.cnt;
            }
        }
        __syncthreads();
        if (l == 0) {
            if constexpr (RMS) {
                // offset 64 (warps 0 + 2, 1 + 3), then 32
                const float t = __fadd_rn(__fadd_rn(xch[0][0], xch[2][0]), __fadd_rn(xch[1][0], xch[3][0]));
                fin[0] = 0.0f;
                fin[1] = finish_rstd(t, Df, p.eps);
            } else {
                Stat g[4];
                for (int w = 0; w < 4; ++w) g[w] = Stat{xch[w][0], xch[w][1], xch[w][2]};
                const Stat f = chan(chan(g[0], g[2]), chan(g[1], g[3]));
                fin[0] = f.mean;
                fin[1] = finish_rstd(f.m2, Df, p.eps);
            }
        }
        __syncthreads();
        const float mean = fin[0], rstd = fin[1];
        const uint16_t *scr = p.scale + b * p.s_scale_b + n * p.s_scale_n;
        const uint16_t *shr = p.shift + b * p.s_shift_b + n * p.s_shift_n;
        uint16_t *orow = p.out + row * D;
        for (int64_t j = l; j < nvec; j += 128)
            for (int e = 0; e < 4; ++e) {
                const int64_t d = 4 * j + e;
                const float v = h_f32<T>(gr ? rr[d] : xr[d * p.sxD]);
                const float y = h_f32<T>(to16_rn<T>(__fmul_rn(rstd, __fsub_rn(v, mean))));
                const float op = h_f32<T>(to16_rn<T>(__fadd_rn(1.0f, h_f32<T>(scr[d]))));
                const float pr = h_f32<T>(to16_rn<T>(__fmul_rn(y, op)));
                const uint16_t o16 = to16_rn<T>(__fadd_rn(pr, h_f32<T>(shr[d])));
                if (p.qscale) {
                    const float q = __fdiv_rn(h_f32<T>(o16), qs);
                    reinterpret_cast<uint8_t *>(p.out)[row * D + d] =
                        (uint8_t)__nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3);
                } else {
                    orow[d] = o16;
                }
            }
        __syncthreads();  // xch / fin are reused by the next row
    }
}

template <DT T, bool RMS>
static cudaError_t run_generic(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    auto k = ln_generic_kernel<T, RMS>;
    const int64_t rows = a.B * a.N;
    const int64_t grid = imin64(rows, (int64_t)dev.sms * blocks_per_sm(k, 128, 0));
    GenericParams p{(uint16_t *)a.out, (const uint16_t *)a.x, a.B, a.N, a.D, a.sxB, a.sxN, a.sxD,
                    (const uint16_t *)a.scale, a.s_scale_b, a.s_scale_n,
                    (const uint16_t *)a.shift, a.s_shift_b, a.s_shift_n, a.eps,
                    (const uint16_t *)a.gate, a.s_gate_b, a.s_gate_n, a.s_gate_d,
                    (const uint16_t *)a.y, (uint16_t *)a.r_out, a.qscale};
    return launch_k(k, dim3((unsigned)grid), dim3(128), 0, s, pdl, p);
}

cudaError_t ln_generic_launch(const LnArgs &a, int dtype, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    if (a.norm == 1)
        return dtype == 0 ? run_generic<DT::BF16, true>(a, pdl, s, dev) : run_generic<DT::FP16, true>(a, pdl, s, dev);
    return dtype == 0 ? run_generic<DT::BF16, false>(a, pdl, s, dev) : run_generic<DT::FP16, false>(a, pdl, s, dev);
}

}  // namespace adaln
