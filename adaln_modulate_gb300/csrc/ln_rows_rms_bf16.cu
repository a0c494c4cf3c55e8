// RMSNorm contiguous-rows kernels, bf16 storage, without a gate.
#include "ln_rows.cuh"

namespace adaln {

cudaError_t rows_rms_bf16(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    return rows_vec<DT::BF16, GATE_NONE, true>(a, pdl, s, dev);
}

}  // namespace adaln
