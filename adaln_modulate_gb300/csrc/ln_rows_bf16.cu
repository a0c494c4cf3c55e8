// ln_modulate contiguous-rows kernels, bf16 storage.
#include "ln_rows.cuh"

namespace adaln {

cudaError_t ln_rows_bf16(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    return rows_vec<DT::BF16, false>(a, RowsGate{}, pdl, s, dev);
}

cudaError_t ln_rows_gate_bf16(const LnArgs &a, const void *y, const void *gate, int64_t s_gate_b, void *r_out,
                            bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    const RowsGate g{(const uint16_t *)y, (const uint16_t *)gate, s_gate_b, (uint16_t *)r_out};
    return rows_vec<DT::BF16, true>(a, g, pdl, s, dev);
}

}  // namespace adaln
