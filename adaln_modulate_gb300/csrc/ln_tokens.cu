// ln_modulate kernels for the transposed view (tokens contiguous) and for
// arbitrary strides.
#include "ln_common.cuh"

namespace adaln {

// ---------------------------------------------------------------------
// tokens contiguous (transposed view): 8 tokens per CTA
// ---------------------------------------------------------------------

constexpr int kTok = 8;

__device__ __forceinline__ void cp_async16_zfill(void *smem, const void *gmem, int src_bytes) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// re-read of a shared-memory slot in the output pass: volatile, so the
// compiler cannot keep the statistics pass's values alive instead
__device__ __forceinline__ void lds16_again(uint32_t *r, const uint4 *p) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}

template <DT T>
__device__ __forceinline__ void push_tokens(f2_t *m, f2_t *q, const uint4 &v, float r) {
    push2(m[0], q[0], f2(lo_f32<T>(v.x), hi_f32<T>(v.x)), r);
    push2(m[1], q[1], f2(lo_f32<T>(v.y), hi_f32<T>(v.y)), r);
    push2(m[2], q[2], f2(lo_f32<T>(v.z), hi_f32<T>(v.z)), r);
    push2(m[3], q[3], f2(lo_f32<T>(v.w), hi_f32<T>(v.w)), r);
}

// chan(lower, upper) on 4 token pairs; `own` is this thread's state
__device__ __forceinline__ void chan_tokens(f2_t *m, f2_t *q, float &cnt, const f2_t *pm,
                                            const f2_t *pq, float pcnt, bool lower) {
    float n;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (lower) {
            chan2(m[k], q[k], cnt, pm[k], pq[k], pcnt, n);
        } else {
            f2_t mm = pm[k], qq = pq[k];
            chan2(mm, qq, pcnt, m[k], q[k], cnt, n);
            m[k] = mm;
            q[k] = qq;
        }
    }
    cnt = n;
}

template <DT T, int NI>
__global__ void __launch_bounds__(128)
ln_tokens_kernel(uint16_t *out, const uint16_t *x, int64_t N, int D, int64_t sxB, int64_t sxD,
                 const uint16_t *scale, int64_t s_scale_b, const uint16_t *shift,
                 int64_t s_shift_b, float eps, int64_t tiles_per_b, int64_t ntiles) {
    extern __shared__ __align__(16) uint4 tile[];  // [NI * 4][128], private per thread
    __shared__ float xch[4][2 * kTok + 1];
    __shared__ float fin[2][kTok];
    const int l = threadIdx.x;
    const int wid = l >> 5;
    const int nvec = D >> 2;
    const float Df = (float)D;
    const float cnt0 = (l < nvec) ? 4.0f * (float)((nvec - 1 - l) / 128 + 1) : 0.0f;
    pdl_wait();

    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int64_t b = t / tiles_per_b;
        const int64_t n0 = (t - b * tiles_per_b) * kTok;
        const int ntok = (int)imin64(kTok, N - n0);
        const uint16_t *xb = x + b * sxB + n0;

        // every thread copies exactly the d-rows of its own logical lane
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            if (128 * i + l < nvec) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int64_t d = 4 * (128 * i + l) + e;
                    cp_async16_zfill(&tile[(i * 4 + e) * 128 + l], xb + d * sxD, 2 * ntok);
                }
            }
            cp_async_commit();
        }

        f2_t m[4], q[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) m[k] = q[k] = f2(0.f, 0.f);
        static_for<0, NI>([&](auto I) {
            constexpr int i = decltype(I)::value;
            cp_async_wait<NI - 1 - i>();
            if (128 * i + l < nvec) {
                static_for<0, 4>([&](auto E) {
                    constexpr int e = decltype(E)::value;
                    const uint4 v = tile[(i * 4 + e) * 128 + l];
                    push_tokens<T>(m, q, v, Rcp<4 * i + e + 1>::value);
                });
            }
        });

        // fold inside the warp: offsets 16, 8, 4, 2, 1
        float cnt = cnt0;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            f2_t pm[4], pq[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                pm[k] = __shfl_xor_sync(0xffffffffu, m[k], off);
                pq[k] = __shfl_xor_sync(0xffffffffu, q[k], off);
            }
            const float pc = __shfl_xor_sync(0xffffffffu, cnt, off);
            chan_tokens(m, q, cnt, pm, pq, pc, (l & off) == 0);
        }
        // offsets 64 then 32 across the four warps
        if ((l & 31) == 0) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                f2_split(m[k], xch[wid][2 * k], xch[wid][2 * k + 1]);
                f2_split(q[k], xch[wid][kTok + 2 * k], xch[wid][kTok + 2 * k + 1]);
            }
            xch[wid][2 * kTok] = cnt;
        }
        __syncthreads();
        if (l < kTok) {
            Stat g[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) g[w] = Stat{xch[w][l], xch[w][kTok + l], xch[w][2 * kTok]};
            const Stat f = chan(chan(g[0], g[2]), chan(g[1], g[3]));
            fin[0][l] = f.mean;
            fin[1][l] = finish_rstd(f.m2, Df, eps);
        }
        __syncthreads();
        f2_t mean2[4], rstd2[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            mean2[k] = f2(fin[0][2 * k], fin[0][2 * k + 1]);
            rstd2[k] = f2(fin[1][2 * k], fin[1][2 * k + 1]);
        }

        // pass 2: this lane's d-rows, 8 tokens each, out rows contiguous in d
        const uint16_t *scr = scale + b * s_scale_b;
        const uint16_t *shr = shift + b * s_shift_b;
        uint16_t *ob = out + (b * N + n0) * (int64_t)D;
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const int j = 128 * i + l;
            if (j < nvec) {
                uint32_t sc[2], sh[2];
                ld_keep8(sc, scr + 4 * j);
                ld_keep8(sh, shr + 4 * j);
                const uint32_t op01 = add16x2<T>(sc[0], one16x2<T>());
                const uint32_t op23 = add16x2<T>(sc[1], one16x2<T>());
                float y[4][kTok];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint32_t w[4];
                    lds16_again(w, &tile[(i * 4 + e) * 128 + l]);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        float xl, xh;
                        unpack_again<T>(w[k], xl, xh);
                        const f2_t u = f2_mul(f2_sub(f2(xl, xh), mean2[k]), rstd2[k]);
                        f2_split(u, y[e][2 * k], y[e][2 * k + 1]);
                    }
                }
#pragma unroll
                for (int tk = 0; tk < kTok; ++tk) {
                    if (tk < ntok) {
                        uint32_t o[2];
                        o[0] = add16x2<T>(mul16x2<T>(pack_rn<T>(y[0][tk], y[1][tk]), op01), sh[0]);
                        o[1] = add16x2<T>(mul16x2<T>(pack_rn<T>(y[2][tk], y[3][tk]), op23), sh[1]);
                        st8(ob + tk * (int64_t)D + 4 * j, o);
                    }
                }
            }
        }
        __syncthreads();  // xch / fin are reused by the next tile
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------
// any strides: one CTA of 128 threads per row, plain binary32 code
// ---------------------------------------------------------------------

template <DT T>
__global__ void __launch_bounds__(128)
ln_generic_kernel(uint16_t *out, const uint16_t *x, int64_t B, int64_t N, int64_t D, int64_t sxB,
                  int64_t sxN, int64_t sxD, const uint16_t *scale, int64_t s_scale_b,
                  const uint16_t *shift, int64_t s_shift_b, float eps) {
    __shared__ float xch[4][3];
    __shared__ float fin[2];
    const int l = threadIdx.x;
    const int64_t nvec = D >> 2;
    const float Df = (float)D;
    pdl_wait();
    for (int64_t row = blockIdx.x; row < B * N; row += gridDim.x) {
        const int64_t b = row / N, n = row - b * N;
        const uint16_t *xr = x + b * sxB + n * sxN;
        Stat s{0.f, 0.f, 0.f};
        for (int64_t j = l; j < nvec; j += 128)
            for (int e = 0; e < 4; ++e) push1(s, h_f32<T>(xr[(4 * j + e) * sxD]));
        for (int off = 16; off >= 1; off >>= 1) s = shfl_stage(s, off);
        if ((l & 31) == 0) {
            xch[l >> 5][0] = s.mean;
            xch[l >> 5][1] = s.m2;
            xch[l >> 5][2] = s.cnt;
        }
        __syncthreads();
        if (l == 0) {
            Stat g[4];
            for (int w = 0; w < 4; ++w) g[w] = Stat{xch[w][0], xch[w][1], xch[w][2]};
            const Stat f = chan(chan(g[0], g[2]), chan(g[1], g[3]));
            fin[0] = f.mean;
            fin[1] = finish_rstd(f.m2, Df, eps);
        }
        __syncthreads();
        const float mean = fin[0], rstd = fin[1];
        const uint16_t *scr = scale + b * s_scale_b, *shr = shift + b * s_shift_b;
        uint16_t *orow = out + row * D;
        for (int64_t d = l; d < D; d += 128) {
            const float v = h_f32<T>(xr[d * sxD]);
            const float y = h_f32<T>(to16_rn<T>(__fmul_rn(rstd, __fsub_rn(v, mean))));
            const float op = h_f32<T>(to16_rn<T>(__fadd_rn(1.0f, h_f32<T>(scr[d]))));
            const float p = h_f32<T>(to16_rn<T>(__fmul_rn(y, op)));
            orow[d] = to16_rn<T>(__fadd_rn(p, h_f32<T>(shr[d])));
        }
        __syncthreads();
    }
    pdl_trigger();
}

template <DT T, int NI>
static cudaError_t run_tokens(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    auto k = ln_tokens_kernel<T, NI>;
    const size_t smem = (size_t)NI * 4 * 128 * sizeof(uint4);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    const int64_t tiles_per_b = (a.N + kTok - 1) / kTok;
    const int64_t ntiles = a.B * tiles_per_b;
    const int64_t grid = imin64(ntiles, (int64_t)dev.sms * blocks_per_sm(k, 128, smem));
    return launch_k(k, dim3((unsigned)grid), dim3(128), smem, s, pdl, (uint16_t *)a.out,
                    (const uint16_t *)a.x, a.N, (int)a.D, a.sxB, a.sxD, (const uint16_t *)a.scale,
                    a.s_scale_b, (const uint16_t *)a.shift, a.s_shift_b, a.eps, tiles_per_b, ntiles);
}

template <DT T>
static cudaError_t tokens_ni(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    switch ((a.D + 511) / 512) {
        case 1: return run_tokens<T, 1>(a, pdl, s, dev);
        case 2: return run_tokens<T, 2>(a, pdl, s, dev);
        case 3: return run_tokens<T, 3>(a, pdl, s, dev);
        case 4: return run_tokens<T, 4>(a, pdl, s, dev);
        case 5: return run_tokens<T, 5>(a, pdl, s, dev);
        case 6: return run_tokens<T, 6>(a, pdl, s, dev);
        case 7: return run_tokens<T, 7>(a, pdl, s, dev);
        case 8: return run_tokens<T, 8>(a, pdl, s, dev);
        case 9: return run_tokens<T, 9>(a, pdl, s, dev);
        case 10: return run_tokens<T, 10>(a, pdl, s, dev);
        case 11: return run_tokens<T, 11>(a, pdl, s, dev);
        case 12: return run_tokens<T, 12>(a, pdl, s, dev);
    }
    return cudaErrorInvalidValue;
}

template <DT T>
static cudaError_t run_generic(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    auto k = ln_generic_kernel<T>;
    const int64_t rows = a.B * a.N;
    const int64_t grid = imin64(rows, (int64_t)dev.sms * blocks_per_sm(k, 128, 0));
    return launch_k(k, dim3((unsigned)grid), dim3(128), 0, s, pdl, (uint16_t *)a.out,
                    (const uint16_t *)a.x, a.B, a.N, a.D, a.sxB, a.sxN, a.sxD,
                    (const uint16_t *)a.scale, a.s_scale_b, (const uint16_t *)a.shift, a.s_shift_b,
                    a.eps);
}

cudaError_t ln_tokens_launch(const LnArgs &a, int dtype, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    return dtype == 0 ? tokens_ni<DT::BF16>(a, pdl, s, dev) : tokens_ni<DT::FP16>(a, pdl, s, dev);
}

cudaError_t ln_generic_launch(const LnArgs &a, int dtype, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    return dtype == 0 ? run_generic<DT::BF16>(a, pdl, s, dev) : run_generic<DT::FP16>(a, pdl, s, dev);
}

}  // namespace adaln
