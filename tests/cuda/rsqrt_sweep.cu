// Test helper (not part of the library): applies CUDA's __frsqrt_rn, the
// 1/sqrt the library's LayerNorm kernels use for rstd, to an array.
#include <cuda_runtime.h>

__global__ void frsqrt_rn_kernel(const float *in, float *out, long long n) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        out[i] = __frsqrt_rn(in[i]);
}

extern "C" int frsqrt_rn_array(const float *in, float *out, long long n) {
    frsqrt_rn_kernel<<<1024, 256>>>(in, out, n);
    return (int)cudaDeviceSynchronize();
}
