// LayerNorm contiguous-rows kernels, bf16 storage, static FP8 (e4m3) output.
#include "ln_rows.cuh"

namespace adaln {

cudaError_t rows_ln_fp8_bf16(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    return rows_vec<DT::BF16, GATE_NONE, false, true>(a, pdl, s, dev);
}

}  // namespace adaln
