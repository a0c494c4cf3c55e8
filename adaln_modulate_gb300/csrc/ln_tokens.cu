// ln_modulate kernels for the transposed view (tokens contiguous) and for
// arbitrary strides.
#include <atomic>

#include "ln_common.cuh"

namespace adaln {

// ---------------------------------------------------------------------
// tokens contiguous (transposed view): 8 tokens per CTA
//
// 256 threads; thread (l, h) is logical lane l = 16*warp + ((tid >> 1) & 15)
// for the tokens 4h .. 4h+3 (h = tid & 1), two f32x2 pairs.  Per tile:
//   1. thread (l, h) copies the d-rows 4*(128*i + l) + 2h + {0, 1} (8
//      tokens, 16 bytes each) into the tile with cp.async; both threads of
//      a lane sit in one warp, so a warp barrier makes the lane's 4 rows
//      visible to both;
//   2. pass 1: serial Welford of lane l for its 4 tokens, states to shared
//      memory;
//   3. warp w folds token w over its 128 lane states (4 lanes per thread in
//      the stride-8 mapping of the contiguous-rows kernel, coefficients from
//      the fold plan); every lane computes the same mean / rstd, lane 0
//      writes them;
//   4. pass 2: thread (l, h) normalises its rows for its 4 tokens, applies
//      the modulate and stores 4 consecutive d of each token (8 bytes).
// Shared-memory reads of a warp cover 256 contiguous bytes (16 lanes x 2
// halves x 8 bytes): two wavefronts, no bank conflict.
// ---------------------------------------------------------------------

constexpr int kTok = 8;
constexpr int kTokThreads = 256;
constexpr int kStPitch = 128 + 24;
static_assert(kTokThreads / 32 == kTok, "one fold warp per token");
__device__ __forceinline__ int st_idx(int l) { return l + 8 * (l >> 5); }


// 8-byte shared load (volatile, so the output pass re-reads the tile rather
// than keeping the statistics pass's values alive)
__device__ __forceinline__ void lds64_again(uint32_t *r, uint32_t saddr) {
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(saddr));
}

template <DT T, int NI>
__global__ void __launch_bounds__(kTokThreads, 2)
ln_tokens_kernel(uint16_t *out, const uint16_t *x, int64_t N, int D, int64_t sxB, int64_t sxD,
                 const uint16_t *scale, int64_t s_scale_b, const uint16_t *shift,
                 int64_t s_shift_b, float eps, int64_t tiles_per_b, int64_t ntiles) {
    extern __shared__ __align__(16) uint4 tile[];   // [NI * 4][128] rows of 8 tokens
    // lane states per token; lane l at l + 8 (l / 32) so that the fold
    // warps' reads (lanes l0 + 8s) hit distinct banks
    __shared__ __align__(16) float st_mean[kTok][kStPitch];
    __shared__ __align__(16) float st_m2[kTok][kStPitch];
    __shared__ float fin[2][kTok];
    __shared__ float plan_s[16][32];  // fold plan of fold-warp thread u, field-major
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int h = tid & 1;
    const int l = warp * 16 + ((tid >> 1) & 15);
    const int nvec = D >> 2;
    const float Df = (float)D;
    const uint32_t tile_s = (uint32_t)__cvta_generic_to_shared(tile);
    // this thread's 8 bytes of the lane-l slot of row group g: tile_s + 16*(g*128 + l) + 8h
    const uint32_t my_s = tile_s + 16 * l + 8 * h;
    pdl_wait();
    pdl_trigger();

    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int64_t b = t / tiles_per_b;
        const int64_t n0 = (t - b * tiles_per_b) * kTok;
        const int ntok = (int)imin64(kTok, N - n0);
        // row d = 4j + e of lane l at step i, j = 128 i + l; this thread
        // copies e = 2h and 2h + 1
        const uint16_t *xl = x + b * sxB + n0 + (int64_t)(4 * l + 2 * h) * sxD;
        const int64_t step_stride = 512 * sxD;

        // 1. copies
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            if (128 * i + l < nvec) {
                const uint16_t *src = xl + i * step_stride;
                cp_async16_zfill(&tile[(i * 4 + 2 * h) * 128 + l], src, 2 * ntok);
                cp_async16_zfill(&tile[(i * 4 + 2 * h + 1) * 128 + l], src + sxD, 2 * ntok);
            }
            cp_async_commit();
        }
        if (t == blockIdx.x && tid < 32) {
            // fold plan of lane-group u = tid (read by every warp in step 3),
            // computed while the first copies are in flight
            const FoldPlan pl = (D % 512 == 0) ? fold_plan_uniform(NI) : fold_plan_runtime(tid, nvec);
            const float *f = reinterpret_cast<const float *>(&pl);
#pragma unroll
            for (int k = 0; k < 16; ++k) plan_s[k][tid] = f[k];
        }

        // 2. pass 1: Welford of lane l, tokens 4h .. 4h+3
        f2_t ma = f2(0.f, 0.f), qa = ma, mb = ma, qb = ma;
        static_for<0, NI>([&](auto I) {
            constexpr int i = decltype(I)::value;
            cp_async_wait<NI - 1 - i>();
            __syncwarp();
            if (128 * i + l < nvec) {
                static_for<0, 4>([&](auto E) {
                    constexpr int e = decltype(E)::value;
                    uint32_t v[2];
                    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                                 : "=r"(v[0]), "=r"(v[1]) : "r"(my_s + 16 * 128 * (i * 4 + e)));
                    constexpr float r = Rcp<4 * i + e + 1>::value;
                    push2(ma, qa, f2(lo_f32<T>(v[0]), hi_f32<T>(v[0])), r);
                    push2(mb, qb, f2(lo_f32<T>(v[1]), hi_f32<T>(v[1])), r);
                });
            }
        });
        {
            const int si = st_idx(l);
            f2_split(ma, st_mean[4 * h][si], st_mean[4 * h + 1][si]);
            f2_split(mb, st_mean[4 * h + 2][si], st_mean[4 * h + 3][si]);
            f2_split(qa, st_m2[4 * h][si], st_m2[4 * h + 1][si]);
            f2_split(qb, st_m2[4 * h + 2][si], st_m2[4 * h + 3][si]);
        }
        // scale / shift of this lane's chunks do not depend on the statistics
        const uint16_t *scr = scale + b * s_scale_b + 4 * l;
        const uint16_t *shr = shift + b * s_shift_b + 4 * l;
        uint32_t sc[NI][2], sh[NI][2];
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            if (128 * i + l < nvec) {
                ld_keep8(sc[i], scr + 512 * i);
                ld_keep8(sh[i], shr + 512 * i);
            }
        }
        __syncthreads();

        // 3. warp w folds token w (a token past the end folds zeros, unused)
        {
            const int u = tid & 31;
            const int i0 = st_idx((u & 7) + 32 * (u >> 3));
            const float *mw = st_mean[warp], *qw = st_m2[warp];
            FoldPlan plan;
            float *f = reinterpret_cast<float *>(&plan);
#pragma unroll
            for (int k = 0; k < 16; ++k) f[k] = plan_s[k][u];
            float mean, m2;
            fold128_s8(f2(mw[i0], mw[i0 + 8]), f2(qw[i0], qw[i0 + 8]), f2(mw[i0 + 16], mw[i0 + 24]),
                       f2(qw[i0 + 16], qw[i0 + 24]), plan, mean, m2);
            const float rstd = finish_rstd(m2, Df, eps);
            if (u == 0) {
                fin[0][warp] = mean;
                fin[1][warp] = rstd;
            }
        }
        __syncthreads();

        // 4. pass 2: tokens 4h .. 4h+3 of lane l
        const f2_t meanA = f2(fin[0][4 * h], fin[0][4 * h + 1]);
        const f2_t meanB = f2(fin[0][4 * h + 2], fin[0][4 * h + 3]);
        const f2_t rstdA = f2(fin[1][4 * h], fin[1][4 * h + 1]);
        const f2_t rstdB = f2(fin[1][4 * h + 2], fin[1][4 * h + 3]);
        uint16_t *ob = out + (b * N + n0 + 4 * h) * (int64_t)D + 4 * l;
        const int nmine = ntok - 4 * h;  // tokens of this half that exist
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            if (128 * i + l < nvec) {
                const uint32_t op01 = add16x2<T>(sc[i][0], one16x2<T>());
                const uint32_t op23 = add16x2<T>(sc[i][1], one16x2<T>());
                float y[4][4];  // [element e of the chunk][token]
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint32_t v[2];
                    lds64_again(v, my_s + 16 * 128 * (i * 4 + e));
                    float x0, x1, x2, x3;
                    unpack_again<T>(v[0], x0, x1);
                    unpack_again<T>(v[1], x2, x3);
                    f2_split(f2_mul(f2_sub(f2(x0, x1), meanA), rstdA), y[e][0], y[e][1]);
                    f2_split(f2_mul(f2_sub(f2(x2, x3), meanB), rstdB), y[e][2], y[e][3]);
                }
#pragma unroll
                for (int tk = 0; tk < 4; ++tk) {
                    if (tk < nmine) {
                        uint32_t o[2];
                        o[0] = add16x2<T>(mul16x2<T>(pack_rn<T>(y[0][tk], y[1][tk]), op01), sh[i][0]);
                        o[1] = add16x2<T>(mul16x2<T>(pack_rn<T>(y[2][tk], y[3][tk]), op23), sh[i][1]);
                        st8(ob + tk * (int64_t)D + 512 * i, o);
                    }
                }
            }
        }
        __syncthreads();  // the tile, st_* and fin are reused by the next tile
    }
}

template <DT T, int NI>
static cudaError_t run_tokens(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    auto k = ln_tokens_kernel<T, NI>;
    const size_t smem = (size_t)NI * 4 * 128 * sizeof(uint4);  // + 8.1 KB static
    static std::atomic<bool> attr_done[64] = {};  // per device, for this (dtype, NI); setting it twice is harmless
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    if (!attr_done[dev.device].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_done[dev.device].store(true, std::memory_order_release);
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

cudaError_t ln_tokens_launch(const LnArgs &a, int dtype, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    if (ln_tokens_tma_fits(a, dev)) {
        const cudaError_t e = ln_tokens_tma_launch(a, dtype, pdl, s, dev);
        if (e != cudaErrorNotSupported) return e;
    }
    return dtype == 0 ? tokens_ni<DT::BF16>(a, pdl, s, dev) : tokens_ni<DT::FP16>(a, pdl, s, dev);
}

}  // namespace adaln
