// adaln_bias_gelu_tanh_noalloc: bias + tanh-GELU without any device
// allocation by this library.
//
// adaln_bias_gelu_tanh keeps its two 65536-entry lookup tables (one per
// storage type) in device memory it allocates with cudaMalloc on first use.
// Some callers cannot let a library allocate: code running under a memory
// arena or pool that owns every byte of the device (a serving process that
// pre-plans all of HBM), code that must not trigger the implicit
// synchronisation of cudaMalloc / cudaFree in the middle of a pipeline, or a
// host program that forbids allocations after start-up.  This entry point
// keeps the same tables in a fixed-size array that is part of the library's
// device image instead, so it never calls cudaMalloc, cudaFree or any
// allocating routine.  The caller still passes (and owns) inputs and output.
//
// Device memory held: kNoallocScratchBytes (256 KiB) on every GPU that
// loads the library, until the process exits.
#include <mutex>

#include "../../include/adaln.h"
#include "kernels.h"

namespace adaln {

constexpr int kTableEntries = 65536;                                   // one per 16-bit pattern
constexpr size_t kNoallocScratchBytes = 2 * kTableEntries * sizeof(uint16_t);  // bf16 + fp16 tables

// The scratch: table of storage type t at element offset t * 65536.
static __device__ __align__(256) uint16_t g_noalloc_scratch[2 * kTableEntries];

namespace {

struct NoallocDev {
    uint16_t *tables = nullptr;  // device address of g_noalloc_scratch on this device
    bool built[2] = {false, false};
};

std::mutex g_mu;
NoallocDev g_state[kApiMaxDevices];

// Both storage types' tables fit the array, whatever the call's rows and
// width: the scratch holds lookup tables, not data of the call.
static_assert(2 * kTableEntries * sizeof(uint16_t) <= kNoallocScratchBytes, "both tables fit");

}  // namespace
}  // namespace adaln

using namespace adaln;

extern "C" adaln_status adaln_bias_gelu_tanh_noalloc(void *out, const void *x, const void *bias,
                                                     int64_t rows, int64_t width, int dtype,
                                                     uint32_t flags, void *stream) {
    // the same argument rules as adaln_bias_gelu_tanh
    adaln_status st = adaln_can_bias_gelu_tanh(out, x, bias, rows, width, dtype, flags);
    if (st != ADALN_OK) return st;
    int dev = 0;
    DeviceInfo info;  // the per-device properties the other entry points use, cached
    if ((st = api_current_device(&dev)) != ADALN_OK || (st = api_device_info(dev, &info)) != ADALN_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    uint16_t *tables = nullptr;
    {
        // set-up, once per device and storage type, with that device current:
        // find the device address of the array, then fill the table on the
        // caller's stream and wait for it
        std::lock_guard<std::mutex> lk(g_mu);
        NoallocDev &d = g_state[dev];
        if (!d.built[dtype]) {
            // the build runs on the caller's stream and is waited for: inside a
            // stream capture it would become part of the caller's graph and the
            // wait would break the capture, so refuse (before any other CUDA
            // call of the set-up) and leave the stream as it is
            cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
            cudaError_t e = cudaStreamIsCapturing(s, &cs);
            if (e != cudaSuccess) return api_cuda_fail(e);
            if (cs != cudaStreamCaptureStatusNone)
                return api_fail_msg(
                    "GELU table of this storage type not set up on this device: make the first "
                    "adaln_bias_gelu_tanh_noalloc call before capturing the stream");
            if (!d.tables) {
                void *p = nullptr;
                e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
                if (e != cudaSuccess) return api_cuda_fail(e);
                d.tables = (uint16_t *)p;
            }
            e = launch_gelu_table_init(d.tables + (size_t)dtype * kTableEntries, dtype, s);
            if (e == cudaSuccess) e = cudaStreamSynchronize(s);
            if (e != cudaSuccess) return api_cuda_fail(e);
            d.built[dtype] = true;
        }
        tables = d.tables;
    }
    GeluArgs a{out, x, bias, rows, width, tables + (size_t)dtype * kTableEntries};
    const cudaError_t e = launch_bias_gelu_tanh(a, dtype, (flags & ADALN_FLAG_PDL) != 0, s, info);
    return e == cudaSuccess ? ADALN_OK : api_cuda_fail(e);
}
