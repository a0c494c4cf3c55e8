// adaln_copy_reference: a same-byte device-to-device copy built like the
// library's streaming kernels (32-byte accesses that bypass L1, a persistent
// grid sized from the SM count and occupancy, programmatic dependent launch
// with the first chunk requested from L2 before the wait).  It is the
// yardstick each op's time is compared against: it moves the bytes an op
// moves with no arithmetic, so "the op takes X % longer than the copy" says
// how much the chain itself costs on this GPU.
#include "../../include/adaln.h"
#include "common.cuh"
#include "kernels.h"

namespace adaln {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;  // 32-byte loads in flight per thread before its stores

__global__ void __launch_bounds__(kCopyThreads)
copy32_kernel(uint8_t *dst, const uint8_t *src, int64_t nvec, int64_t tail) {
    if (threadIdx.x == 0) {
        const int64_t v0 = (int64_t)blockIdx.x * kCopyThreads;
        const int64_t v1 = imin64(v0 + kCopyThreads, nvec);
        if (v1 > v0) prefetch_l2(src + 32 * v0, (uint64_t)(v1 - v0) * 32);
    }
    pdl_wait();
    pdl_trigger();
    const int64_t stride = (int64_t)gridDim.x * kCopyThreads;
    for (int64_t v = (int64_t)blockIdx.x * kCopyThreads + threadIdx.x; v < nvec; v += kCopyUnroll * stride) {
        uint32_t r[kCopyUnroll][8];
#pragma unroll
        for (int k = 0; k < kCopyUnroll; ++k)
            if (v + k * stride < nvec) ld_stream32(r[k], src + 32 * (v + k * stride));
#pragma unroll
        for (int k = 0; k < kCopyUnroll; ++k)
            if (v + k * stride < nvec) st32(dst + 32 * (v + k * stride), r[k]);
    }
    // the last bytes % 32, one byte per thread of the first CTA
    if (blockIdx.x == 0 && threadIdx.x < tail) dst[32 * nvec + threadIdx.x] = src[32 * nvec + threadIdx.x];
}

}  // namespace adaln

using namespace adaln;

extern "C" adaln_status adaln_copy_reference(void *dst, const void *src, int64_t bytes, uint32_t flags,
                                             void *stream) {
    if (!dst || !src) return ADALN_E_NULL;
    if (flags & ~ADALN_FLAG_PDL) return ADALN_E_VALUE;
    if (bytes < 1 || bytes > ((int64_t)1 << 46)) return ADALN_E_SHAPE;
    if (((uintptr_t)dst | (uintptr_t)src) & 31u) return ADALN_E_ALIGN;
    const uintptr_t d = (uintptr_t)dst, s = (uintptr_t)src;
    if (d < s + (uintptr_t)bytes && s < d + (uintptr_t)bytes) return ADALN_E_OVERLAP;
    int dev = 0;
    DeviceInfo info;
    adaln_status st;
    if ((st = api_current_device(&dev)) != ADALN_OK || (st = api_device_info(dev, &info)) != ADALN_OK) return st;
    const int64_t nvec = bytes / 32, tail = bytes % 32;
    auto k = copy32_kernel;
    const int64_t grid = imin64((int64_t)info.sms * blocks_per_sm(k, kCopyThreads, 0),
                                imin64((nvec + kCopyThreads - 1) / kCopyThreads, (int64_t)1 << 30));
    const cudaError_t e = launch_k(k, dim3((unsigned)(grid > 0 ? grid : 1)), dim3(kCopyThreads), 0,
                                   (cudaStream_t)stream, (flags & ADALN_FLAG_PDL) != 0, (uint8_t *)dst,
                                   (const uint8_t *)src, nvec, tail);
    return e == cudaSuccess ? ADALN_OK : api_cuda_fail(e);
}
