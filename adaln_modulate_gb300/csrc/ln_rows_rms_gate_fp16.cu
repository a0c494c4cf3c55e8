// RMSNorm contiguous-rows kernels, fp16 storage, with the residual gate-add in front.
#include "ln_rows.cuh"

namespace adaln {

cudaError_t rows_rms_gate_fp16(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    return rows_gated<DT::FP16, true>(a, pdl, s, dev);
}

}  // namespace adaln
