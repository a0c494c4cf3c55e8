// Test helper (not part of the library): the quotient helper the static FP8
// quantisers use (div_by_recip, Markstein's correction from RN(1/b)) and
// CUDA's __fdiv_rn, side by side, on an array of numerators; and the rows
// kernel's 4-wide e4m3 quantisers on arrays of 16-bit storage values (the
// form the kernel picks for the scale, or one forced).
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

// form: 0 the one the rows kernel picks (plain product if the CTA's check
// passes, else the branch-free correction for an ordinary scale, else the
// window), 1 the window, 2 the branch-free correction (for an ordinary scale)
template <adaln::DT T>
__global__ void quant4_kernel(const uint32_t *y, float qs, uint32_t *codes, long long nq, int form, int memo,
                              int *picked) {
    adaln::QuantE4M3 c = adaln::quant_setup<T>(qs);
    __shared__ unsigned long long memo_s;
    if (threadIdx.x == 0) memo_s = memo ? adaln::plain_memo_load<T>() : 0ull;
    __syncthreads();
    adaln::quant_pick_plain<T>(c, &memo_s, threadIdx.x, blockDim.x);
    if (blockIdx.x == 0 && threadIdx.x == 0) *picked = (c.fast ? 1 : 0) | (c.plain ? 2 : 0);
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < nq;
         i += (long long)gridDim.x * blockDim.x)
        codes[i] = form == 1   ? adaln::quant4_e4m3_window<T>(y + 2 * i, c)
                   : form == 2 ? adaln::quant4_e4m3_fast<T>(y + 2 * i, c)
                               : adaln::quant4_e4m3<T>(y + 2 * i, c);
}

// y: 4 * nq storage values (bf16 when fp16 == 0), codes: 4 * nq bytes;
// memo != 0: consult and update the device memo of the multiplier search
// (as the rows kernel does), else always search; *picked (device int): bit
// 0 the branch-free correction applies to qs, bit 1 the plain product does
extern "C" int quant4_sweep(const void *y, float qs, void *codes, long long nq, int fp16, int form, int memo,
                            void *picked) {
    if (fp16)
        quant4_kernel<adaln::DT::FP16><<<1024, 256>>>((const uint32_t *)y, qs, (uint32_t *)codes, nq, form, memo,
                                                       (int *)picked);
    else
        quant4_kernel<adaln::DT::BF16><<<1024, 256>>>((const uint32_t *)y, qs, (uint32_t *)codes, nq, form, memo,
                                                       (int *)picked);
    return (int)cudaDeviceSynchronize();
}
