// ln_modulate for the transposed view (tokens contiguous), tiles of 16
// tokens loaded by the tensor memory accelerator.
//
// x is read through a 4-D tensor map {N, nvec, 4, B}: token n, chunk j,
// element e of the chunk (d = 4 j + e) and sample b.  A tile is 16 tokens of
// one sample; step i of the lane DAG (chunks 128 i .. 128 i + 127) is one
// box {16, 128, 4, 1} of 16 KB with its own mbarrier, so pass 1 of step i
// starts as soon as its box has landed while later boxes are in flight.  The
// box lands as [e][j][16 tokens]: 32 contiguous bytes (one full sector) per
// d-row in global memory, and in shared memory the rows of one e-plane sit
// 32 bytes apart, so a warp reading lanes 8w .. 8w+7 for one e spreads over
// every bank (two wavefronts for 256 bytes).  Chunks past D/4 and tokens
// past N are outside the tensor and arrive as zeros.
//
// Thread (l, h), l = tid / 2 the logical lane and h = tid % 2, owns tokens
// 8h .. 8h+7 of lane l and reads 16 bytes of each of its four d-rows per
// step (a warp reads 512 contiguous bytes).  Per tile: pass 1 (serial
// Welford of lane l for 8 tokens, four f32x2 chains) -> lane states in
// shared memory -> warp w folds tokens 2w and 2w+1 and writes mean / rstd ->
// pass 2 normalises, modulates with op = round(1 + scale) and shift from a
// per-sample shared table, and stores 8 bytes per token.
//
// 256 threads of at most 128 registers and about 111 KB of shared memory for
// D <= 2560, so two CTAs fit on an SM: with programmatic dependent launch the
// next call's CTAs become resident while this call's still run, and each
// asks L2 for its first tile before it waits for this grid to finish, so its
// tile is mostly in L2 by the time it may load it.  The next tile of a CTA
// that loops over several is prefetched into L2 while the current one runs.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "../../include/adaln.h"
#include "ln_common.cuh"

namespace adaln {

constexpr int kTT = 16;             // tokens per tile
constexpr int kTTThreads = 256;     // (128 lanes) x (2 token groups of 8)
constexpr int kTTRowBytes = kTT * 2;
constexpr int kStepBytes = 512 * kTTRowBytes;   // one box: 128 chunks x 4 elements x 16 tokens
constexpr int kPlaneBytes = 128 * kTTRowBytes;  // one e-plane of a box
constexpr int kTTPitch = 154;       // lane-state row pitch: 4 * pitch = 8 (mod 32) banks
constexpr int kWaitSpins = 1 << 22; // bounded mbarrier waits
constexpr int kTTMaxNI = 10;        // D <= 5120
constexpr int kFillPer = (kTTMaxNI * 512 / 2 + kTTThreads - 1) / kTTThreads;  // table pairs per thread
constexpr int kTTWarps = kTTThreads / 32;
static_assert(2 * kTTWarps == kTT, "two fold tokens per warp");

// Timed-out mbarrier waits of the TMA tile kernel on this device (should stay 0).
__device__ unsigned int g_tma_wait_timeouts;

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// true once the phase with this parity has completed; false after kWaitSpins polls
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (int it = 0; it < kWaitSpins; ++it) {
        uint32_t done;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap *map, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global [%0, {%1, %2, %3, %4}];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}

template <DT T, int NI>
__global__ void __launch_bounds__(kTTThreads, 2)
ln_tokens_tma_kernel(const __grid_constant__ CUtensorMap tmx, uint16_t *out, int64_t N, int D,
                     const uint16_t *scale, int64_t s_scale_b, const uint16_t *shift, int64_t s_shift_b,
                     float eps, int64_t tiles_per_b, int64_t ntiles) {
    extern __shared__ unsigned char tt_dyn[];  // [1 KB alignment slack][tile][op/shift table]
    __shared__ __align__(16) float st_mean[kTT][kTTPitch];
    __shared__ __align__(16) float st_m2[kTT][kTTPitch];
    __shared__ float fin[2][kTT];
    __shared__ float plan_s[16][32];
    __shared__ __align__(8) uint64_t bar[NI];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int l = tid >> 1;
    const int h = tid & 1;
    const int nvec = D >> 2;
    const float Df = (float)D;
    const uint32_t dyn_s = (uint32_t)__cvta_generic_to_shared(tt_dyn);
    const uint32_t tile_s = (dyn_s + 1023u) & ~1023u;  // [step][e][chunk][16 tokens]
    uint32_t *opsh = reinterpret_cast<uint32_t *>(tt_dyn + (tile_s - dyn_s) + NI * kStepBytes);
    const uint32_t bar_s = (uint32_t)__cvta_generic_to_shared(&bar[0]);
    const uint32_t my_s = tile_s + (uint32_t)(kTTRowBytes * l + 16 * h);  // (step 0, e 0) of this thread

    // Launch parameters are not data of the previous kernel: read them, fetch
    // the tensor map's descriptor, set up the barriers and arm them with the
    // first tile's byte counts before waiting on that kernel (the first read
    // of a parameter misses the constant cache, about a microsecond; an armed
    // phase still completes only once its bytes have arrived).  Thread 0
    // keeps the first tile's coordinates in registers and issues its loads
    // as the first thing after the wait (anything ahead of them there, such
    // as a parameter read or a 64-bit division, delays the whole landing);
    // the other threads take the coordinates from shared memory.
    __shared__ int64_t first_tile[2];
    int b0 = 0, f0 = 0;  // the first tile (thread 0)
    if (tid == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmx)) : "memory");
#pragma unroll
        for (int i = 0; i < NI; ++i) mbar_init(bar_s + 8 * i, 1);
#pragma unroll
        for (int i = 0; i < NI; ++i) mbar_expect_tx(bar_s + 8 * i, (uint32_t)kStepBytes);
        asm volatile("fence.mbarrier_init.release.cluster;\nfence.proxy.async.shared::cta;" ::: "memory");
        b0 = (int)((int64_t)blockIdx.x / tiles_per_b);
        f0 = (int)(((int64_t)blockIdx.x - (int64_t)b0 * tiles_per_b) * kTT);
        first_tile[0] = b0;
        first_tile[1] = f0;
        // Ask L2 for the first tile and its sample's scale / shift rows now,
        // while the previous kernel may still be running.  A prefetch is only
        // a hint with no effect on what later loads return: L2 is where every
        // SM's accesses to global memory meet, so the loads issued after the
        // wait still see everything the previous kernel wrote.
#pragma unroll
        for (int i = 0; i < NI; ++i) tma_prefetch_4d(&tmx, f0, 128 * i, 0, b0);
        prefetch_l2(scale + b0 * s_scale_b, (uint64_t)D * 2);
        prefetch_l2(shift + b0 * s_shift_b, (uint64_t)D * 2);
    }
    __syncthreads();
    pdl_wait();
    if (tid == 0) {
        // the first tile's loads, from one thread in box order (boxes issued
        // by several warps at once land interleaved, the first one late)
#pragma unroll
        for (int i = 0; i < NI; ++i)
            tma_load_4d(tile_s + (uint32_t)(i * kStepBytes), &tmx, f0, 128 * i, 0, b0, bar_s + 8 * i);
    }
    pdl_trigger();

    int64_t table_b = -1;
    uint32_t parity = 0;
    int64_t b = first_tile[0], n0 = first_tile[1];
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, parity ^= 1u) {
        if (t != blockIdx.x) {
            b = t / tiles_per_b;
            n0 = (t - b * tiles_per_b) * kTT;
        }

        if (tid == 0) {
            if (t != blockIdx.x) {
                // the previous tile's shared reads are ordered before these
                // asynchronous writes by the barrier that ended it
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
#pragma unroll
                for (int i = 0; i < NI; ++i) {
                    mbar_expect_tx(bar_s + 8 * i, (uint32_t)kStepBytes);
                    tma_load_4d(tile_s + (uint32_t)(i * kStepBytes), &tmx, (int)n0, 128 * i, 0, (int)b, bar_s + 8 * i);
                }
            }
            const int64_t tn = t + gridDim.x;
            if (tn < ntiles) {
                const int64_t bn = tn / tiles_per_b;
                const int nn0 = (int)((tn - bn * tiles_per_b) * kTT);
#pragma unroll
                for (int i = 0; i < NI; ++i) tma_prefetch_4d(&tmx, nn0, 128 * i, 0, (int)bn);
            }
        }
        // op = round(1 + scale) and shift of sample b, interleaved per column
        // pair: loaded now (they land with the boxes), stored after pass 1
        const bool new_table = b != table_b;
        uint32_t s2[kFillPer], h2[kFillPer];
        if (new_table) {
#pragma unroll
            for (int k = 0; k < kFillPer; ++k) {
                const int e = tid + k * kTTThreads;
                if (e < D / 2) {
                    asm("ld.global.nc.b32 %0, [%1];" : "=r"(s2[k]) : "l"(scale + b * s_scale_b + 2 * e));
                    asm("ld.global.nc.b32 %0, [%1];" : "=r"(h2[k]) : "l"(shift + b * s_shift_b + 2 * e));
                }
            }
        }
        if (t == blockIdx.x && warp == kTTWarps - 1) {
            // fold plan of lane group u (read by every fold warp), while the boxes land
            const int u = tid & 31;
            const FoldPlan pl = (D % 512 == 0) ? fold_plan_uniform(NI) : fold_plan_runtime(u, nvec);
            const float *f = reinterpret_cast<const float *>(&pl);
#pragma unroll
            for (int k = 0; k < 16; ++k) plan_s[k][u] = f[k];
        }

        // pass 1: Welford of lane l for the token pairs (8h + 2k, 8h + 2k + 1)
        bool ok = true;
        f2_t m[4], q[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) m[k] = q[k] = f2(0.f, 0.f);
        static_for<0, NI>([&](auto I) {
            constexpr int i = decltype(I)::value;
            ok = mbar_wait(bar_s + 8 * i, parity) && ok;
            if (128 * i + l < nvec) {
                static_for<0, 4>([&](auto E) {
                    constexpr int e = decltype(E)::value;
                    uint32_t v[4];
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                                 : "r"(my_s + (uint32_t)(i * kStepBytes + e * kPlaneBytes)));
                    constexpr float r = Rcp<4 * i + e + 1>::value;
#pragma unroll
                    for (int k = 0; k < 4; ++k) push2(m[k], q[k], f2(lo_f32<T>(v[k]), hi_f32<T>(v[k])), r);
                });
            }
        });
        {
            const int si = l + 8 * (l >> 5);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                f2_split(m[k], st_mean[8 * h + 2 * k][si], st_mean[8 * h + 2 * k + 1][si]);
                f2_split(q[k], st_m2[8 * h + 2 * k][si], st_m2[8 * h + 2 * k + 1][si]);
            }
        }
        if (new_table) {
#pragma unroll
            for (int k = 0; k < kFillPer; ++k) {
                const int e = tid + k * kTTThreads;
                if (e < D / 2) {
                    opsh[2 * e] = add16x2<T>(s2[k], one16x2<T>());
                    opsh[2 * e + 1] = h2[k];
                }
            }
            table_b = b;
        }
        if (!__syncthreads_and(ok)) {
            // a box never arrived: count it, give the copies another bounded
            // wait so none is left writing into this CTA, and stop
            if (tid == 0) atomicAdd(&g_tma_wait_timeouts, 1u);
#pragma unroll
            for (int i = 0; i < NI; ++i) mbar_wait(bar_s + 8 * i, parity);
            return;
        }

        // warp w folds tokens 2w and 2w + 1 together, one f32x2 lane per token
        // (a token past N folds zeros and is not stored)
        {
            const int u = tid & 31;
            const int i0 = (u & 7) + 32 * (u >> 3) + 8 * (u >> 3);
            FoldPlan plan;
            float *f = reinterpret_cast<float *>(&plan);
#pragma unroll
            for (int k = 0; k < 16; ++k) f[k] = plan_s[k][u];
            const float *mA = st_mean[2 * warp], *qA = st_m2[2 * warp];
            const float *mB = st_mean[2 * warp + 1], *qB = st_m2[2 * warp + 1];
            f2_t mean2, m22;
            fold128_s8_x2(f2(mA[i0], mB[i0]), f2(qA[i0], qB[i0]), f2(mA[i0 + 8], mB[i0 + 8]),
                          f2(qA[i0 + 8], qB[i0 + 8]), f2(mA[i0 + 16], mB[i0 + 16]), f2(qA[i0 + 16], qB[i0 + 16]),
                          f2(mA[i0 + 24], mB[i0 + 24]), f2(qA[i0 + 24], qB[i0 + 24]), plan, mean2, m22);
            float meanA, meanB, m2A, m2B;
            f2_split(mean2, meanA, meanB);
            f2_split(m22, m2A, m2B);
            const float rstdA = finish_rstd(m2A, Df, eps), rstdB = finish_rstd(m2B, Df, eps);
            if (u == 0) {
                fin[0][2 * warp] = meanA;
                fin[1][2 * warp] = rstdA;
                fin[0][2 * warp + 1] = meanB;
                fin[1][2 * warp + 1] = rstdB;
            }
        }
        __syncthreads();

        // pass 2: tokens 8h .. 8h+7 of lane l
        f2_t mean2[4], rstd2[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            mean2[k] = f2(fin[0][8 * h + 2 * k], fin[0][8 * h + 2 * k + 1]);
            rstd2[k] = f2(fin[1][8 * h + 2 * k], fin[1][8 * h + 2 * k + 1]);
        }
        const int nmine = (int)imin64(8, N - n0 - 8 * h);  // tokens of this group inside N
        uint16_t *ob = out + (b * N + n0 + 8 * h) * (int64_t)D + 4 * l;
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            if (128 * i + l < nvec) {
                const uint4 os = *reinterpret_cast<const uint4 *>(opsh + 4 * (128 * i + l));
                float y[4][8];  // [element e of the chunk][token]
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint32_t v[4];
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                                 : "r"(my_s + (uint32_t)(i * kStepBytes + e * kPlaneBytes)));
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        float xa, xb;
                        unpack_again<T>(v[k], xa, xb);
                        f2_split(f2_mul(f2_sub(f2(xa, xb), mean2[k]), rstd2[k]), y[e][2 * k], y[e][2 * k + 1]);
                    }
                }
#pragma unroll
                for (int tk = 0; tk < 8; ++tk) {
                    if (tk < nmine) {
                        uint32_t o[2];
                        o[0] = add16x2<T>(mul16x2<T>(pack_rn<T>(y[0][tk], y[1][tk]), os.x), os.y);
                        o[1] = add16x2<T>(mul16x2<T>(pack_rn<T>(y[2][tk], y[3][tk]), os.z), os.w);
                        st8(ob + tk * (int64_t)D + 512 * i, o);
                    }
                }
            }
        }
        __syncthreads();  // the tile, lane states, fin and the table are reused by the next tile
    }
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

constexpr size_t kStaticSmemBound = 24 * 1024;  // lane states, fin, plan, barriers (< 21 KB)

size_t tma_dyn_smem(int64_t D) {
    const int64_t ni = (D + 511) / 512;
    return 1024 + (size_t)ni * kStepBytes + (size_t)D * 4;
}

template <DT T, int NI>
cudaError_t run_tokens_tma(const LnArgs &a, const CUtensorMap &map, bool pdl, cudaStream_t s,
                           const DeviceInfo &dev) {
    auto k = ln_tokens_tma_kernel<T, NI>;
    const size_t smem = tma_dyn_smem(a.D);
    static std::atomic<bool> attr_done[64] = {};  // per device; setting it twice is harmless
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    if (!attr_done[dev.device].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)tma_dyn_smem(NI * 512));
        if (e != cudaSuccess) return e;
        attr_done[dev.device].store(true, std::memory_order_release);
    }
    const int64_t tiles_per_b = (a.N + kTT - 1) / kTT;
    const int64_t ntiles = a.B * tiles_per_b;
    const int64_t grid = imin64(ntiles, (int64_t)dev.sms * blocks_per_sm(k, kTTThreads, smem));
    return launch_k(k, dim3((unsigned)grid), dim3(kTTThreads), smem, s, pdl, map, (uint16_t *)a.out, a.N,
                    (int)a.D, (const uint16_t *)a.scale, a.s_scale_b, (const uint16_t *)a.shift, a.s_shift_b,
                    a.eps, tiles_per_b, ntiles);
}

template <DT T>
cudaError_t tma_ni(const LnArgs &a, const CUtensorMap &map, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    switch ((a.D + 511) / 512) {
        case 1: return run_tokens_tma<T, 1>(a, map, pdl, s, dev);
        case 2: return run_tokens_tma<T, 2>(a, map, pdl, s, dev);
        case 3: return run_tokens_tma<T, 3>(a, map, pdl, s, dev);
        case 4: return run_tokens_tma<T, 4>(a, map, pdl, s, dev);
        case 5: return run_tokens_tma<T, 5>(a, map, pdl, s, dev);
        case 6: return run_tokens_tma<T, 6>(a, map, pdl, s, dev);
        case 7: return run_tokens_tma<T, 7>(a, map, pdl, s, dev);
        case 8: return run_tokens_tma<T, 8>(a, map, pdl, s, dev);
        case 9: return run_tokens_tma<T, 9>(a, map, pdl, s, dev);
        case 10: return run_tokens_tma<T, 10>(a, map, pdl, s, dev);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

bool ln_tokens_tma_fits(const LnArgs &a, const DeviceInfo &dev) {
    return (a.D + 511) / 512 <= kTTMaxNI && a.N <= INT32_MAX && a.D <= INT32_MAX && a.B <= INT32_MAX &&
           tma_dyn_smem(a.D) + kStaticSmemBound <= (size_t)dev.max_smem_optin;
}

namespace {

// The tensor map of x: dims {token, chunk j, element e, sample}, d = 4 j + e.
bool encode_x_map(const LnArgs &a, CUtensorMap *map) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc) return false;
    const int64_t sxB_bytes = (a.B == 1 ? a.D * a.sxD : a.sxB) * 2;
    const cuuint64_t gdim[4] = {(cuuint64_t)a.N, (cuuint64_t)(a.D / 4), 4, (cuuint64_t)a.B};
    const cuuint64_t gstride[3] = {(cuuint64_t)(4 * a.sxD * 2), (cuuint64_t)(a.sxD * 2), (cuuint64_t)sxB_bytes};
    const cuuint32_t box[4] = {(cuuint32_t)kTT, 128, 4, 1};
    const cuuint32_t estride[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void *>(a.x), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// The TMA tile kernel takes these arguments: the tile fits in shared memory
// and the driver builds the tensor map (host-side only, no device work).
bool ln_tokens_tma_ready(const LnArgs &a, const DeviceInfo &dev) {
    CUtensorMap map;
    return ln_tokens_tma_fits(a, dev) && encode_x_map(a, &map);
}

// Encodes the tensor map of x and launches; cudaErrorNotSupported when the
// map cannot be built (the caller then uses the cp.async tile kernel).
cudaError_t ln_tokens_tma_launch(const LnArgs &a, int dtype, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    CUtensorMap map;
    if (!encode_x_map(a, &map)) return cudaErrorNotSupported;
    return dtype == 0 ? tma_ni<DT::BF16>(a, map, pdl, s, dev) : tma_ni<DT::FP16>(a, map, pdl, s, dev);
}

}  // namespace adaln

extern "C" adaln_status adaln_tma_wait_timeouts(uint32_t *count) {
    if (!count) return ADALN_E_NULL;
    const cudaError_t e = cudaMemcpyFromSymbol(count, adaln::g_tma_wait_timeouts, sizeof(uint32_t));
    return e == cudaSuccess ? ADALN_OK : ADALN_E_CUDA;
}
