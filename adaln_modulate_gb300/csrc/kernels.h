// Host-side launchers of the sm_103a kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/adaln.h"

namespace adaln {

struct DeviceInfo {
    int device = -1;
    int sms = 0;
    int max_smem_optin = 0;
    int l2_bytes = 0;
};

// One norm + modulate call: out = norm(v) * (1 + scale) + shift with v = x,
// or v = x + gate * y (written to r_out) when gate is set.  The fields after
// eps default to LayerNorm with one scale / shift row per sample and no gate.
struct LnArgs {
    void *out;
    const void *x;
    int64_t B, N, D, sxB, sxN, sxD;
    const void *scale;
    int64_t s_scale_b;
    const void *shift;
    int64_t s_shift_b;
    float eps;
    int64_t s_scale_n = 0, s_shift_n = 0;  // per-token operand rows (0: one row per sample)
    int norm = 0;                          // 0 LayerNorm, 1 RMSNorm (both without affine)
    const void *gate = nullptr;            // residual gate (b, n, d) at b*s_gate_b + n*s_gate_n + d*s_gate_d
    int64_t s_gate_b = 0, s_gate_n = 0, s_gate_d = 1;
    const void *y = nullptr;               // with a gate: y and r_out contiguous (B, N, D), x too
    void *r_out = nullptr;
    const float *qscale = nullptr;         // set: out is e4m3 bytes, e4m3(y / *qscale) (static FP8)
};

struct QkArgs {
    void *q_out;
    const void *q;
    int64_t rows_q;
    void *k_out;
    const void *k;
    int64_t rows_k;
    int64_t Dh;
    const void *wq, *bq, *wk, *bk;  // RMSNorm: bq, bk unused
    float eps;
    bool rms = false;               // per-head RMSNorm with a weight instead of LayerNorm with affine
};

struct GateArgs {
    void *out;
    const void *x;
    const void *gate;
    int64_t s_gate_b;
    const void *y;
    int64_t B, N, D;
};

// out_k = table[k] + temb[:, :, k] as K contiguous binary32 slices
// (dtypes: 0 bf16, 1 fp16, 2 binary32)
struct TembArgs {
    void *out;        // slice k at out + k * s_out_k (floats), each (B, S, D)
    int64_t s_out_k;
    const void *table;  // (K, D)
    int table_dtype;
    const void *temb;   // (B, S, K, D)
    int temb_dtype;
    int64_t B, S, K, D;
};

struct GeluArgs {
    void *out;
    const void *x;
    const void *bias;
    int64_t rows, width;
    const void *table;  // 65536 storage values of the dtype
};

// Which ln_modulate kernel a call takes (exposed for tests and the bench).
enum LnPath : int { LN_PATH_ROWS = 0, LN_PATH_TOKENS = 1, LN_PATH_GENERIC = 2, LN_PATH_TOKENS_TMA = 3 };
int ln_modulate_path(const LnArgs &a);

cudaError_t launch_ln_modulate(const LnArgs &a, int dtype, bool pdl, cudaStream_t s,
                               const DeviceInfo &dev);
// the transposed-view tile kernel fed by tensor-memory-accelerator boxes
bool ln_tokens_tma_fits(const LnArgs &a, const DeviceInfo &dev);
bool ln_tokens_tma_ready(const LnArgs &a, const DeviceInfo &dev);
cudaError_t ln_tokens_tma_launch(const LnArgs &a, int dtype, bool pdl, cudaStream_t s, const DeviceInfo &dev);
cudaError_t launch_qk_head_layernorm(const QkArgs &a, int dtype, bool pdl, cudaStream_t s,
                                     const DeviceInfo &dev);
cudaError_t launch_residual_gate_add(const GateArgs &a, int dtype, bool pdl, cudaStream_t s,
                                     const DeviceInfo &dev);
// norm + modulate with every option of LnArgs (RMSNorm, per-token rows, a
// residual gate); launch_ln_modulate is the same call
cudaError_t launch_norm_scale_shift(const LnArgs &a, int dtype, bool pdl, cudaStream_t s, const DeviceInfo &dev);
cudaError_t launch_bias_gelu_tanh(const GeluArgs &a, int dtype, bool pdl, cudaStream_t s,
                                  const DeviceInfo &dev);
cudaError_t launch_gelu_table_init(void *table, int dtype, cudaStream_t s);
cudaError_t launch_temb_table_slices(const TembArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev);

// cudaLaunchKernelEx with the optional programmatic-dependent-launch attribute
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     bool pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Host helpers of the C ABI (api.cu) for entry points defined in other
// files: the current device (an ordinal past the library's 64 per-device
// slots is an error with its own text), its cached properties, and the text
// that adaln_last_cuda_error() returns after a failure (a CUDA error, or a
// message of the caller's).  Each returns ADALN_OK or ADALN_E_CUDA.
adaln_status api_current_device(int *dev);
adaln_status api_device_info(int dev, DeviceInfo *out);
adaln_status api_cuda_fail(cudaError_t e);
adaln_status api_fail_msg(const char *msg);
constexpr int kApiMaxDevices = 64;

// Resident blocks per SM of a kernel at a block size / dynamic smem, cached
// per (kernel, block size, smem); every device this library drives is the
// same model.
int blocks_per_sm_cached(const void *kernel, int threads, size_t smem);

template <typename K>
int blocks_per_sm(K kernel, int threads, size_t smem) {
    return blocks_per_sm_cached(reinterpret_cast<const void *>(kernel), threads, smem);
}

}  // namespace adaln
