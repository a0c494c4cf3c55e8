// Test helper (not part of the library): the quotient helper the static FP8
// quantisers use (div_by_recip, Markstein's correction from RN(1/b)) and
// CUDA's __fdiv_rn, side by side, on an array of numerators; and the rows
// kernel's 4-wide e4m3 quantisers on arrays of 16-bit storage values (the
// form the kernel picks for the scale, or the window form for any scale).
#include <cuda_runtime.h>

#include "../../adaln_modulate_gb300/csrc/quant_e4m3.cuh"

__global__ void div_sweep_kernel(const float *a, float b, float *mine, float *ieee, long long n) {
    const float r = __frcp_rn(b);
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        mine[i] = adaln::div_by_recip(a[i], b, r);
        ieee[i] = __fdiv_rn(a[i], b);
    }
}

extern "C" int div_sweep(const float *a, float b, float *mine, float *ieee, long long n) {
    div_sweep_kernel<<<1024, 256>>>(a, b, mine, ieee, n);
    return (int)cudaDeviceSynchronize();
}

template <adaln::DT T>
__global__ void quant4_kernel(const uint32_t *y, float qs, uint32_t *codes, long long nq, int window,
                              int *fast) {
    const adaln::QuantE4M3 c = adaln::quant_setup<T>(qs);
    if (blockIdx.x == 0 && threadIdx.x == 0) *fast = c.fast ? 1 : 0;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < nq;
         i += (long long)gridDim.x * blockDim.x)
        codes[i] = window ? adaln::quant4_e4m3_window<T>(y + 2 * i, c) : adaln::quant4_e4m3<T>(y + 2 * i, c);
}

// y: 4 * nq storage values (bf16 when fp16 == 0), codes: 4 * nq bytes;
// window != 0 forces the window form; *fast (device int) tells whether the
// branch-free form applies to qs
extern "C" int quant4_sweep(const void *y, float qs, void *codes, long long nq, int fp16, int window, void *fast) {
    if (fp16)
        quant4_kernel<adaln::DT::FP16><<<1024, 256>>>((const uint32_t *)y, qs, (uint32_t *)codes, nq, window,
                                                       (int *)fast);
    else
        quant4_kernel<adaln::DT::BF16><<<1024, 256>>>((const uint32_t *)y, qs, (uint32_t *)codes, nq, window,
                                                       (int *)fast);
    return (int)cudaDeviceSynchronize();
}
