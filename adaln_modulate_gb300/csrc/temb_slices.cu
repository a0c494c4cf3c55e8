// temb_table_slices for sm_103a: the K modulation chunks of a per-token
// (B, S, K, D) temb, each added to its table row and written to its own
// contiguous binary32 (B, S, D) slice in one pass.
//
// Follows the "temb_table_slices" entry of the SGLang Diffusion "Fused
// Kernels" page (adaLN modulation and gating table, and its note: the eager
// (scale_shift_table + temb.float()).chunk(6, dim=2) materialises the full
// binary32 sum and hands six strided slices downstream, whose .contiguous()
// copies it again; here every output byte is written once, already
// contiguous).  Per element: out = float(table[k, d]) + float(temb[b, s, k, d])
// (one IEEE binary32 addition; the promotions are exact).
//
// Mapping: a persistent grid walks temb in storage order, 8 consecutive d
// of one (token, chunk) row per thread and step (16-byte bf16 / fp16 or
// 32-byte binary32 loads, one 32-byte store to slice k); the table (K x D,
// at most a few hundred KB) stays in L1 / L2.  Shapes or pointers that do
// not allow the 8-wide accesses take the scalar kernel.
#include "common.cuh"
#include "kernels.h"

namespace adaln {

constexpr int kTembThreads = 256;

// 8 consecutive values of a bf16 / fp16 (16 bytes) or binary32 (32 bytes)
// array as binary32
template <int DTY>
__device__ __forceinline__ void load8_f32(float *v, const void *p, bool keep) {
    if constexpr (DTY == 2) {
        uint32_t r[8];
        if (keep) ld_keep32(r, p); else ld_stream32(r, p);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
    } else {
        uint32_t r[4];
        if (keep) ld_keep16(r, p); else ld_stream16(r, p);
        constexpr DT T = DTY == 0 ? DT::BF16 : DT::FP16;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = lo_f32<T>(r[i]);
            v[2 * i + 1] = hi_f32<T>(r[i]);
        }
    }
}

template <int DTY>
__device__ __forceinline__ float load1_f32(const void *p, int64_t i) {
    if constexpr (DTY == 2) return static_cast<const float *>(p)[i];
    constexpr DT T = DTY == 0 ? DT::BF16 : DT::FP16;
    return h_f32<T>(static_cast<const uint16_t *>(p)[i]);
}

// VEC: 8 elements per thread and step (D % 8 == 0, aligned pointers and
// slice stride); otherwise one element
template <int TDT, int EDT, bool VEC>
__global__ void __launch_bounds__(kTembThreads)
temb_slices_kernel(float *__restrict__ out, int64_t s_out_k, const void *__restrict__ table,
                   const void *__restrict__ temb, int64_t BS, int64_t K, int64_t D) {
    const int64_t W = VEC ? D / 8 : D;  // units per (token, chunk) row
    const int64_t total = BS * K * W;
    const int64_t stride = (int64_t)gridDim.x * kTembThreads;
    // unit u = (bs * K + k) * W + w (temb storage order): (bs, k, w) advanced
    // by the grid step with carries, no division per iteration
    const int64_t u0 = (int64_t)blockIdx.x * kTembThreads + threadIdx.x;
    const int64_t qr = stride / W, rw = stride - qr * W;      // rows and units of one step
    const int64_t qs0 = qr / K, rk0 = qr - qs0 * K;           // a step of qr rows
    const int64_t qs1 = (qr + 1) / K, rk1 = (qr + 1) - qs1 * K;  // a step of qr + 1 rows
    int64_t row0 = u0 / W, w = u0 - row0 * W;
    int64_t bs = row0 / K, k = row0 - bs * K;
    // (the divisions above depend on launch parameters only)
    pdl_wait();
    pdl_trigger();
    for (int64_t u = u0; u < total; u += stride) {
        const int64_t row = bs * K + k;
        if constexpr (VEC) {
            const int64_t d = 8 * w;
            float e[8], t[8];
            load8_f32<EDT>(e, static_cast<const char *>(temb) + (row * D + d) * (EDT == 2 ? 4 : 2), false);
            load8_f32<TDT>(t, static_cast<const char *>(table) + (k * D + d) * (TDT == 2 ? 4 : 2), true);
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = __float_as_uint(__fadd_rn(t[i], e[i]));
            st32(out + k * s_out_k + bs * D + d, o);
        } else {
            out[k * s_out_k + bs * D + w] = __fadd_rn(load1_f32<TDT>(table, k * D + w), load1_f32<EDT>(temb, row * D + w));
        }
        w += rw;
        const bool carry = w >= W;
        if (carry) w -= W;
        bs += carry ? qs1 : qs0;
        k += carry ? rk1 : rk0;
        if (k >= K) {
            k -= K;
            ++bs;
        }
    }
}

template <int TDT, int EDT, bool VEC>
static cudaError_t run_temb(const TembArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    auto k = temb_slices_kernel<TDT, EDT, VEC>;
    const int64_t units = a.B * a.S * a.K * (VEC ? a.D / 8 : a.D);
    const int64_t grid = imin64((units + kTembThreads - 1) / kTembThreads,
                                (int64_t)dev.sms * blocks_per_sm(k, kTembThreads, 0));
    return launch_k(k, dim3((unsigned)grid), dim3(kTembThreads), 0, s, pdl, (float *)a.out, a.s_out_k, a.table,
                    a.temb, a.B * a.S, a.K, a.D);
}

static bool al(const void *p, int a) { return ((uintptr_t)p % (uintptr_t)a) == 0; }

template <int TDT, int EDT>
static cudaError_t temb_vec(const TembArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    const int te = TDT == 2 ? 4 : 2, ee = EDT == 2 ? 4 : 2;
    const bool vec = a.D % 8 == 0 && a.s_out_k % 8 == 0 && al(a.out, 32) && al(a.table, 8 * te) &&
                     al(a.temb, 8 * ee);
    return vec ? run_temb<TDT, EDT, true>(a, pdl, s, dev) : run_temb<TDT, EDT, false>(a, pdl, s, dev);
}

template <int TDT>
static cudaError_t temb_e(const TembArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    switch (a.temb_dtype) {
        case 0: return temb_vec<TDT, 0>(a, pdl, s, dev);
        case 1: return temb_vec<TDT, 1>(a, pdl, s, dev);
        case 2: return temb_vec<TDT, 2>(a, pdl, s, dev);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_temb_table_slices(const TembArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    switch (a.table_dtype) {
        case 0: return temb_e<0>(a, pdl, s, dev);
        case 1: return temb_e<1>(a, pdl, s, dev);
        case 2: return temb_e<2>(a, pdl, s, dev);
    }
    return cudaErrorInvalidValue;
}

}  // namespace adaln
