// ln_modulate kernels for the transposed view (tokens contiguous) and for
// arbitrary strides.
#include "ln_common.cuh"

namespace adaln {

// ---------------------------------------------------------------------
// tokens contiguous (transposed view): 8 tokens per CTA
//
// 512 threads; thread (l, p) is logical lane l = 8*warp + ((tid >> 2) & 7)
// for the token pair p = tid & 3 (tokens 2p, 2p+1).  Data flow per tile:
//   1. thread (l, p) copies the d-rows 4*(128*i + l) + p (8 tokens, 16 bytes
//      each) into the tile with cp.async; the 4 threads of a lane sit in one
//      warp, so a warp barrier makes a lane's 4 rows visible to all of them;
//   2. pass 1: serial Welford of lane l for tokens 2p, 2p+1 (one f32x2 op
//      covers both tokens), state to shared memory;
//   3. warps 0..7 fold token t = warp over the 128 lane states (4 lanes per
//      thread in the stride-8 mapping of the contiguous-rows kernel, with
//      the combine coefficients precomputed) and write mean / rstd;
//   4. pass 2: thread (l, p) normalises its rows for its two tokens, applies
//      the modulate and stores 4 consecutive d of each token (8 bytes).
// Shared-memory reads of a warp cover 128 contiguous bytes (8 lanes x 4
// token pairs x 4 bytes), so they are free of bank conflicts.
// ---------------------------------------------------------------------

constexpr int kTok = 8;
constexpr int kTokThreads = 512;
constexpr int kStPitch = 128 + 24;
__device__ __forceinline__ int st_idx(int l) { return l + 8 * (l >> 5); }

__device__ __forceinline__ void cp_async16_zfill(void *smem, const void *gmem, int src_bytes) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint32_t lds32(const void *p) {
    uint32_t r;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(r) : "r"((uint32_t)__cvta_generic_to_shared(p)));
    return r;
}

template <DT T, int NI>
__global__ void __launch_bounds__(kTokThreads, 2)
ln_tokens_kernel(uint16_t *out, const uint16_t *x, int64_t N, int D, int64_t sxB, int64_t sxD,
                 const uint16_t *scale, int64_t s_scale_b, const uint16_t *shift,
                 int64_t s_shift_b, float eps, int64_t tiles_per_b, int64_t ntiles) {
    extern __shared__ __align__(16) uint4 tile[];   // [NI * 4][128] rows of 8 tokens
    // lane states per token; lane l at l + 8 (l / 32) so that the fold
    // warps' reads (lanes l0 + 8s) hit 32 distinct banks
    __shared__ __align__(16) float st_mean[kTok][kStPitch];
    __shared__ __align__(16) float st_m2[kTok][kStPitch];
    __shared__ float fin[2][kTok];
    __shared__ float plan_s[16][32];  // fold coefficients of fold-warp thread u, field-major
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int p = tid & 3;
    const int l = warp * 8 + ((tid >> 2) & 7);
    const int nvec = D >> 2;
    const float Df = (float)D;
    const unsigned char *tb = reinterpret_cast<const unsigned char *>(tile);
    if (tid < 32) {
        const FoldPlan pl = (D % 512 == 0) ? fold_plan_uniform(NI) : fold_plan_runtime(tid, nvec);
        const float *f = reinterpret_cast<const float *>(&pl);
#pragma unroll
        for (int k = 0; k < 16; ++k) plan_s[k][tid] = f[k];
    }
    pdl_wait();

    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int64_t b = t / tiles_per_b;
        const int64_t n0 = (t - b * tiles_per_b) * kTok;
        const int ntok = (int)imin64(kTok, N - n0);
        const uint16_t *xb = x + b * sxB + n0;

        // 1. this thread's share of the lane's rows: element e = p of each chunk
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            if (128 * i + l < nvec) {
                const int64_t d = 4 * (128 * i + l) + p;
                cp_async16_zfill(&tile[(i * 4 + p) * 128 + l], xb + d * sxD, 2 * ntok);
            }
            cp_async_commit();
        }

        // 2. pass 1: Welford of lane l, tokens 2p and 2p+1
        f2_t m = f2(0.f, 0.f), q = m;
        static_for<0, NI>([&](auto I) {
            constexpr int i = decltype(I)::value;
            cp_async_wait<NI - 1 - i>();
            __syncwarp();
            if (128 * i + l < nvec) {
                static_for<0, 4>([&](auto E) {
                    constexpr int e = decltype(E)::value;
                    const uint32_t v = *reinterpret_cast<const uint32_t *>(
                        tb + 16 * ((i * 4 + e) * 128 + l) + 4 * p);
                    push2(m, q, f2(lo_f32<T>(v), hi_f32<T>(v)), Rcp<4 * i + e + 1>::value);
                });
            }
        });
        f2_split(m, st_mean[2 * p][st_idx(l)], st_mean[2 * p + 1][st_idx(l)]);
        f2_split(q, st_m2[2 * p][st_idx(l)], st_m2[2 * p + 1][st_idx(l)]);
        // scale / shift of this lane's chunks do not depend on the statistics
        const uint16_t *scr = scale + b * s_scale_b;
        const uint16_t *shr = shift + b * s_shift_b;
        uint32_t sc[NI][2], sh[NI][2];
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const int j = 128 * i + l;
            if (j < nvec) {
                ld_keep8(sc[i], scr + 4 * j);
                ld_keep8(sh[i], shr + 4 * j);
            }
        }
        __syncthreads();

        // 3. warp w < 8 folds token w over the 128 lanes (stride-8 mapping)
        if (warp < kTok) {
            const int u = tid & 31;
            const int i0 = st_idx((u & 7) + 32 * (u >> 3));
            const float *sm = st_mean[warp], *sq = st_m2[warp];
            FoldPlan plan;
            float *f = reinterpret_cast<float *>(&plan);
#pragma unroll
            for (int k = 0; k < 16; ++k) f[k] = plan_s[k][u];
            float mean, m2;
            fold128_s8(f2(sm[i0], sm[i0 + 8]), f2(sq[i0], sq[i0 + 8]), f2(sm[i0 + 16], sm[i0 + 24]),
                       f2(sq[i0 + 16], sq[i0 + 24]), plan, mean, m2);
            if (u == 0) {
                fin[0][warp] = mean;
                fin[1][warp] = finish_rstd(m2, Df, eps);
            }
        }
        __syncthreads();

        // 4. pass 2: tokens 2p, 2p+1 of lane l
        const f2_t mean2 = f2(fin[0][2 * p], fin[0][2 * p + 1]);
        const f2_t rstd2 = f2(fin[1][2 * p], fin[1][2 * p + 1]);
        uint16_t *ob = out + (b * N + n0) * (int64_t)D;
        const bool st0 = 2 * p < ntok, st1 = 2 * p + 1 < ntok;
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const int j = 128 * i + l;
            if (j < nvec) {
                const uint32_t op01 = add16x2<T>(sc[i][0], one16x2<T>());
                const uint32_t op23 = add16x2<T>(sc[i][1], one16x2<T>());
                float y0[4], y1[4];  // token 2p / 2p+1, element e of the chunk
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t v = lds32(tb + 16 * ((i * 4 + e) * 128 + l) + 4 * p);
                    float xl, xh;
                    unpack_again<T>(v, xl, xh);
                    f2_split(f2_mul(f2_sub(f2(xl, xh), mean2), rstd2), y0[e], y1[e]);
                }
                uint32_t o[2];
                if (st0) {
                    o[0] = add16x2<T>(mul16x2<T>(pack_rn<T>(y0[0], y0[1]), op01), sh[i][0]);
                    o[1] = add16x2<T>(mul16x2<T>(pack_rn<T>(y0[2], y0[3]), op23), sh[i][1]);
                    st8(ob + (2 * p) * (int64_t)D + 4 * j, o);
                }
                if (st1) {
                    o[0] = add16x2<T>(mul16x2<T>(pack_rn<T>(y1[0], y1[1]), op01), sh[i][0]);
                    o[1] = add16x2<T>(mul16x2<T>(pack_rn<T>(y1[2], y1[3]), op23), sh[i][1]);
                    st8(ob + (2 * p + 1) * (int64_t)D + 4 * j, o);
                }
            }
        }
        __syncthreads();  // the tile, st_* and fin are reused by the next tile
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
    const size_t smem = (size_t)NI * 4 * 128 * sizeof(uint4);  // + 8.1 KB static
    static bool attr_done[64] = {};  // per device, for this (dtype, NI)
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    if (!attr_done[dev.device]) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_done[dev.device] = true;
    }
    const int64_t tiles_per_b = (a.N + kTok - 1) / kTok;
    const int64_t ntiles = a.B * tiles_per_b;
    const int64_t grid = imin64(ntiles, (int64_t)dev.sms * blocks_per_sm(k, kTokThreads, smem));
    return launch_k(k, dim3((unsigned)grid), dim3(kTokThreads), smem, s, pdl, (uint16_t *)a.out,
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
