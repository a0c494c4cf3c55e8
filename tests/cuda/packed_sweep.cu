// Test helper (not part of the library): every pair of 16-bit operands
// through the packed add / multiply the kernels use for the modulate, gate
// and bias steps (add16x2 / mul16x2 of common.cuh), against the same
// operation in binary32 followed by one round-to-nearest-even conversion to
// the storage type.  That conversion is written here from the IEEE 754
// definition in integer arithmetic; the hardware conversion (cvt.rn) is
// checked against it on every binary32 result as well.  NaN matches NaN.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../adaln_modulate_gb300/csrc/common.cuh"

using adaln::DT;

// binary32 -> bf16, round to nearest even; NaN -> 0x7FC0 (sign kept)
__device__ __forceinline__ uint32_t rne_bf16(uint32_t u) {
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return ((u >> 16) & 0x8000u) | 0x7FC0u;
    return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

// binary32 -> fp16, round to nearest even, subnormal results kept, overflow
// to infinity; NaN -> 0x7E00 (sign kept)
__device__ __forceinline__ uint32_t rne_f16(uint32_t u) {
    const uint32_t sign = (u >> 16) & 0x8000u, a = u & 0x7FFFFFFFu;
    if (a > 0x7F800000u) return sign | 0x7E00u;
    if (a >= 0x477FF000u) return sign | 0x7C00u;        // >= 65520 rounds to infinity
    if (a >= 0x38800000u) {                              // normal fp16 range (>= 2^-14)
        uint32_t r = (a - 0x38000000u) >> 13;            // rebias 127 -> 15, keep 10 fraction bits
        const uint32_t rem = a & 0x1FFFu;
        r += (rem > 0x1000u) || (rem == 0x1000u && (r & 1u));
        return sign | r;                                 // a carry into the exponent is correct
    }
    if (a <= 0x33000000u) return sign;                   // <= 2^-25 (half the smallest subnormal; ties to 0)
    const uint32_t e = a >> 23, m = (a & 0x7FFFFFu) | 0x800000u;
    const uint32_t sh = 126u - e;                        // value = m * 2^(e - 150), unit 2^-24
    uint32_t r = m >> sh;
    const uint32_t rem = m & ((1u << sh) - 1u), half = 1u << (sh - 1u);
    r += (rem > half) || (rem == half && (r & 1u));
    return sign | r;
}

__device__ __forceinline__ bool nan16(uint32_t h, bool f16) {
    return f16 ? ((h & 0x7C00u) == 0x7C00u && (h & 0x3FFu)) : ((h & 0x7F80u) == 0x7F80u && (h & 0x7Fu));
}
__device__ __forceinline__ bool same16(uint32_t x, uint32_t y, bool f16) {
    const bool nx = nan16(x, f16), ny = nan16(y, f16);
    return (nx || ny) ? (nx && ny) : x == y;
}

template <DT T, bool MUL>
__global__ void packed_sweep_kernel(unsigned long long *res) {
    constexpr bool F16 = T == DT::FP16;
    unsigned long long bad = 0, bad_cvt = 0;
    // pair index q covers (a, b) and (a, b + 1): a = q >> 15, b = 2 (q & 0x7FFF)
    for (uint64_t q = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; q < (1ull << 31);
         q += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t a = (uint32_t)(q >> 15), b = (uint32_t)(q & 0x7FFFu) * 2u;
        const uint32_t pa = a | (a << 16), pb = b | ((b + 1u) << 16);
        const uint32_t got = MUL ? adaln::mul16x2<T>(pa, pb) : adaln::add16x2<T>(pa, pb);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float fa = adaln::lo_f32<T>(a), fb = adaln::lo_f32<T>(b + (uint32_t)k);
            const float r = MUL ? __fmul_rn(fa, fb) : __fadd_rn(fa, fb);
            const uint32_t u = __float_as_uint(r);
            const uint32_t want = F16 ? rne_f16(u) : rne_bf16(u);
            const uint32_t hw = adaln::to16_rn<T>(r);
            const uint32_t g = (got >> (16 * k)) & 0xFFFFu;
            if (!same16(g, want, F16)) {
                ++bad;
                atomicMin(&res[2], (unsigned long long)a << 16 | (b + k));
            }
            if (!same16(hw, want, F16)) ++bad_cvt;
        }
    }
    if (bad) atomicAdd(&res[0], bad);
    if (bad_cvt) atomicAdd(&res[1], bad_cvt);
}

// op 0 add, 1 mul; fp16 0 bf16, 1 fp16.  out: [mismatches of the packed op,
// mismatches of cvt.rn against the integer rounding, first bad (a << 16 | b)]
extern "C" int packed_sweep(int op, int fp16, unsigned long long *out) {
    unsigned long long *res = nullptr;
    if (cudaMalloc(&res, 3 * sizeof(unsigned long long)) != cudaSuccess) return -1;
    const unsigned long long init[3] = {0, 0, ~0ull};
    cudaMemcpy(res, init, sizeof(init), cudaMemcpyHostToDevice);
    const dim3 g(152 * 8), b(256);
    if (op == 0 && !fp16) packed_sweep_kernel<DT::BF16, false><<<g, b>>>(res);
    if (op == 1 && !fp16) packed_sweep_kernel<DT::BF16, true><<<g, b>>>(res);
    if (op == 0 && fp16) packed_sweep_kernel<DT::FP16, false><<<g, b>>>(res);
    if (op == 1 && fp16) packed_sweep_kernel<DT::FP16, true><<<g, b>>>(res);
    int e = (int)cudaDeviceSynchronize();
    cudaMemcpy(out, res, 3 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    cudaFree(res);
    return e;
}
