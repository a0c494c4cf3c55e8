// Streaming chains for sm_103a: residual gate-add and bias + tanh-GELU.
//
// residual_gate_add follows the "Fused Kernels" page (adaLN modulation and
// gating table: residual + gate * update, bit-exact) as wired for GLM-Image
// in PR #34008: out = round(x + round(gate * y)).
//
// bias_gelu_tanh follows PR #37075 ("功能与动机" and the bias_gelu_tanh
// kernel): v = round(fp32(x) + fp32(bias)) to the storage type, then
// tanh-GELU, rounded again.  On this GPU the activation is a lookup: a
// 65536-entry table (one per storage type) holds round(G(v)) for every
// 16-bit pattern v, built once per device by gelu_table_kernel and staged
// into shared memory by every CTA of the persistent streaming kernel.
//
// One add or multiply of two storage values done by the packed 16-bit
// instructions equals binary32 arithmetic followed by one storage rounding
// (see add16x2 in common.cuh), which is what the chains specify.
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace adaln {

// elements of one thread-iteration: 16 (32-byte accesses), 8, 4
template <int EPT> struct Acc;
template <> struct Acc<16> {
    static __device__ __forceinline__ void ld_s(uint32_t *r, const uint16_t *p) { ld_stream32(r, p); }
    static __device__ __forceinline__ void ld_k(uint32_t *r, const uint16_t *p) { ld_keep32(r, p); }
    static __device__ __forceinline__ void st(uint16_t *p, const uint32_t *r) { st32(p, r); }
};
template <> struct Acc<8> {
    static __device__ __forceinline__ void ld_s(uint32_t *r, const uint16_t *p) { ld_stream16(r, p); }
    static __device__ __forceinline__ void ld_k(uint32_t *r, const uint16_t *p) { ld_keep16(r, p); }
    static __device__ __forceinline__ void st(uint16_t *p, const uint32_t *r) { st16(p, r); }
};
template <> struct Acc<4> {
    static __device__ __forceinline__ void ld_s(uint32_t *r, const uint16_t *p) { ld_stream8(r, p); }
    static __device__ __forceinline__ void ld_k(uint32_t *r, const uint16_t *p) { ld_keep8(r, p); }
    static __device__ __forceinline__ void st(uint16_t *p, const uint32_t *r) { st8(p, r); }
};

// ------------------------------------------------------------ gate add

constexpr int kEwThreads = 512;

template <DT T, int EPT>
__global__ void __launch_bounds__(kEwThreads)
gate_add_kernel(uint16_t *out, const uint16_t *x, const uint16_t *gate, int64_t s_gate_b,
                const uint16_t *y, int64_t nvec, int64_t ND, int64_t D) {
    // ask L2 for this CTA's first x and y elements before waiting on the
    // previous kernel (a hint only: loads after the wait still see its writes)
    if (threadIdx.x == 0) {
        const int64_t e0 = (int64_t)blockIdx.x * kEwThreads * EPT;
        const int64_t e1 = imin64(e0 + (int64_t)kEwThreads * EPT, nvec * EPT);
        if (e1 > e0) {
            prefetch_l2(x + e0, (uint64_t)(e1 - e0) * 2);
            prefetch_l2(y + e0, (uint64_t)(e1 - e0) * 2);
        }
    }
    constexpr int R = EPT / 2;
    const int64_t stride = (int64_t)gridDim.x * kEwThreads;
    // sample b and column col of the thread's element, advanced by the
    // grid step with a carry (no division per iteration); the divisions
    // depend on launch parameters only and are done before the wait
    const int64_t v0 = (int64_t)blockIdx.x * kEwThreads + threadIdx.x, step = stride * EPT;
    const int64_t qb = step / ND, rb = step - qb * ND, rc = step % D;
    int64_t b = v0 * EPT / ND, in_b = v0 * EPT - b * ND, col = v0 * EPT % D;
    pdl_wait();
    pdl_trigger();
    for (int64_t v = v0; v < nvec; v += stride) {
        const int64_t e0 = v * EPT;
        uint32_t xr[R], yr[R], gr[R], o[R];
        Acc<EPT>::ld_s(xr, x + e0);
        Acc<EPT>::ld_s(yr, y + e0);
        Acc<EPT>::ld_k(gr, gate + b * s_gate_b + col);
#pragma unroll
        for (int k = 0; k < R; ++k) o[k] = add16x2<T>(xr[k], mul16x2<T>(gr[k], yr[k]));
        Acc<EPT>::st(out + e0, o);
        b += qb;
        in_b += rb;
        if (in_b >= ND) {
            in_b -= ND;
            ++b;
        }
        col += rc;
        if (col >= D) col -= D;
    }
}

// any D / alignment: one element per thread-iteration in binary32
template <DT T>
__global__ void __launch_bounds__(kEwThreads)
gate_add_scalar_kernel(uint16_t *out, const uint16_t *x, const uint16_t *gate, int64_t s_gate_b,
                       const uint16_t *y, int64_t n, int64_t ND, int64_t D) {
    pdl_wait();
    pdl_trigger();
    const int64_t stride = (int64_t)gridDim.x * kEwThreads;
    const int64_t e_0 = (int64_t)blockIdx.x * kEwThreads + threadIdx.x;
    const int64_t qb = stride / ND, rb = stride - qb * ND, rc = stride % D;
    int64_t b = e_0 / ND, in_b = e_0 - b * ND, col = e_0 % D;
    for (int64_t e = e_0; e < n; e += stride, b += qb, in_b += rb, col += rc) {
        if (in_b >= ND) {
            in_b -= ND;
            ++b;
        }
        if (col >= D) col -= D;
        const float gy = h_f32<T>(to16_rn<T>(__fmul_rn(h_f32<T>(gate[b * s_gate_b + col]), h_f32<T>(y[e]))));
        out[e] = to16_rn<T>(__fadd_rn(h_f32<T>(x[e]), gy));
    }
}

static bool al(const void *p, int a) { return ((uintptr_t)p % (uintptr_t)a) == 0; }

template <DT T, int EPT>
static cudaError_t run_gate(const GateArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    const int64_t n = a.B * a.N * a.D;
    if constexpr (EPT == 1) {
        auto k = gate_add_scalar_kernel<T>;
        const int64_t grid = imin64((n + kEwThreads - 1) / kEwThreads,
                                          (int64_t)dev.sms * blocks_per_sm(k, kEwThreads, 0));
        return launch_k(k, dim3((unsigned)grid), dim3(kEwThreads), 0, s, pdl, (uint16_t *)a.out,
                        (const uint16_t *)a.x, (const uint16_t *)a.gate, a.s_gate_b,
                        (const uint16_t *)a.y, n, a.N * a.D, a.D);
    } else {
        auto k = gate_add_kernel<T, EPT>;
        const int64_t nvec = n / EPT;
        const int64_t grid = imin64((nvec + kEwThreads - 1) / kEwThreads,
                                          (int64_t)dev.sms * blocks_per_sm(k, kEwThreads, 0));
        return launch_k(k, dim3((unsigned)grid), dim3(kEwThreads), 0, s, pdl, (uint16_t *)a.out,
                        (const uint16_t *)a.x, (const uint16_t *)a.gate, a.s_gate_b,
                        (const uint16_t *)a.y, nvec, a.N * a.D, a.D);
    }
}

template <DT T>
static cudaError_t gate_dispatch(const GateArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    for (int ept : {16, 8, 4}) {
        const int vb = 2 * ept;
        if (a.D % ept == 0 && al(a.out, vb) && al(a.x, vb) && al(a.y, vb) && al(a.gate, vb) &&
            (a.B == 1 || a.s_gate_b % ept == 0)) {
            if (ept == 16) return run_gate<T, 16>(a, pdl, s, dev);
            if (ept == 8) return run_gate<T, 8>(a, pdl, s, dev);
            return run_gate<T, 4>(a, pdl, s, dev);
        }
    }
    return run_gate<T, 1>(a, pdl, s, dev);
}

cudaError_t launch_residual_gate_add(const GateArgs &a, int dtype, bool pdl, cudaStream_t s,
                                     const DeviceInfo &dev) {
    return dtype == 0 ? gate_dispatch<DT::BF16>(a, pdl, s, dev) : gate_dispatch<DT::FP16>(a, pdl, s, dev);
}

// ----------------------------------------------------------- GELU table

// table[h] = round16(rn_f32(G(v))) with v the value of pattern h and
// G(v) = 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))), evaluated in
// binary64 as v / (1 + exp(-2 z)) (the same real number, free of the
// cancellation in 1 + tanh(z) for z << 0).  G(+inf) = +inf, G(-inf) = NaN.
template <DT T>
__global__ void gelu_table_kernel(uint16_t *table) {
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= 65536) return;
    const float vf = h_f32<T>((uint16_t)h);
    float g;
    if (isnan(vf)) {
        g = vf;
    } else if (isinf(vf)) {
        g = vf > 0.0f ? vf : __int_as_float(0x7fc00000);
    } else {
        const double v = (double)vf;
        const double k0 = 0.79788456080286535587989211986876;  // sqrt(2/pi)
        const double k1 = 0.044715;
        const double z = __dmul_rn(k0, __dadd_rn(v, __dmul_rn(k1, __dmul_rn(v, __dmul_rn(v, v)))));
        const double den = __dadd_rn(1.0, exp(__dmul_rn(-2.0, z)));
        g = __double2float_rn(__ddiv_rn(v, den));
    }
    table[h] = to16_rn<T>(g);
}

cudaError_t launch_gelu_table_init(void *table, int dtype, cudaStream_t s) {
    if (dtype == 0)
        gelu_table_kernel<DT::BF16><<<256, 256, 0, s>>>((uint16_t *)table);
    else
        gelu_table_kernel<DT::FP16><<<256, 256, 0, s>>>((uint16_t *)table);
    return cudaGetLastError();
}

// ---------------------------------------------------------- bias + GELU

constexpr int kGeluThreads = 1024;
constexpr size_t kGeluSmem = 65536 * sizeof(uint16_t);

template <DT T>
__device__ __forceinline__ uint32_t gelu2(const uint16_t *tab, uint32_t v) {
    const uint32_t lo = tab[v & 0xffffu];
    const uint32_t hi = tab[v >> 16];
    return lo | (hi << 16);
}

template <DT T, int EPT>
__global__ void __launch_bounds__(kGeluThreads, 1)
bias_gelu_kernel(uint16_t *out, const uint16_t *x, const uint16_t *bias, int64_t nvec, int64_t width,
                 const uint16_t *table) {
    extern __shared__ __align__(16) uint16_t tab[];
    constexpr int R = EPT / 2;
    // the table is written once per device before any launch: stage it
    // before waiting on the preceding grid
    for (int i = threadIdx.x; i < 65536 / 8; i += kGeluThreads)
        reinterpret_cast<uint4 *>(tab)[i] = reinterpret_cast<const uint4 *>(table)[i];
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    const int64_t stride = (int64_t)gridDim.x * kGeluThreads;
    for (int64_t v = (int64_t)blockIdx.x * kGeluThreads + threadIdx.x; v < nvec; v += stride) {
        const int64_t e0 = v * EPT;
        const int64_t col = e0 % width;
        uint32_t xr[R], br[R], o[R];
        Acc<EPT>::ld_s(xr, x + e0);
        Acc<EPT>::ld_k(br, bias + col);
#pragma unroll
        for (int k = 0; k < R; ++k) o[k] = gelu2<T>(tab, add16x2<T>(xr[k], br[k]));
        Acc<EPT>::st(out + e0, o);
    }
}

template <DT T>
__global__ void __launch_bounds__(kEwThreads)
bias_gelu_scalar_kernel(uint16_t *out, const uint16_t *x, const uint16_t *bias, int64_t n,
                        int64_t width, const uint16_t *table) {
    pdl_wait();
    pdl_trigger();
    const int64_t stride = (int64_t)gridDim.x * kEwThreads;
    for (int64_t e = (int64_t)blockIdx.x * kEwThreads + threadIdx.x; e < n; e += stride) {
        const uint16_t v = to16_rn<T>(__fadd_rn(h_f32<T>(x[e]), h_f32<T>(bias[e % width])));
        out[e] = table[v];
    }
}

template <DT T, int EPT>
static cudaError_t run_gelu(const GeluArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    const int64_t n = a.rows * a.width;
    if constexpr (EPT == 1) {
        auto k = bias_gelu_scalar_kernel<T>;
        const int64_t grid = imin64((n + kEwThreads - 1) / kEwThreads,
                                          (int64_t)dev.sms * blocks_per_sm(k, kEwThreads, 0));
        return launch_k(k, dim3((unsigned)grid), dim3(kEwThreads), 0, s, pdl, (uint16_t *)a.out,
                        (const uint16_t *)a.x, (const uint16_t *)a.bias, n, a.width,
                        (const uint16_t *)a.table);
    } else {
        auto k = bias_gelu_kernel<T, EPT>;
        static std::atomic<bool> attr_set[64] = {};  // per device; setting it twice is harmless
        if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
        if (!attr_set[dev.device].load(std::memory_order_acquire)) {
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGeluSmem);
            if (e != cudaSuccess) return e;
            attr_set[dev.device].store(true, std::memory_order_release);
        }
        const int64_t nvec = n / EPT;
        const int64_t grid = imin64((nvec + kGeluThreads - 1) / kGeluThreads,
                                          (int64_t)dev.sms * blocks_per_sm(k, kGeluThreads, kGeluSmem));
        return launch_k(k, dim3((unsigned)grid), dim3(kGeluThreads), kGeluSmem, s, pdl,
                        (uint16_t *)a.out, (const uint16_t *)a.x, (const uint16_t *)a.bias, nvec, a.width,
                        (const uint16_t *)a.table);
    }
}

template <DT T>
static cudaError_t gelu_dispatch(const GeluArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    for (int ept : {16, 8, 4}) {
        const int vb = 2 * ept;
        if (a.width % ept == 0 && al(a.out, vb) && al(a.x, vb) && al(a.bias, vb)) {
            if (ept == 16) return run_gelu<T, 16>(a, pdl, s, dev);
            if (ept == 8) return run_gelu<T, 8>(a, pdl, s, dev);
            return run_gelu<T, 4>(a, pdl, s, dev);
        }
    }
    return run_gelu<T, 1>(a, pdl, s, dev);
}

cudaError_t launch_bias_gelu_tanh(const GeluArgs &a, int dtype, bool pdl, cudaStream_t s,
                                  const DeviceInfo &dev) {
    return dtype == 0 ? gelu_dispatch<DT::BF16>(a, pdl, s, dev) : gelu_dispatch<DT::FP16>(a, pdl, s, dev);
}

}  // namespace adaln
