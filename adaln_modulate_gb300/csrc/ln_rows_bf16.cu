// ln_modulate contiguous-rows kernel, bf16 storage.
#include "ln_rows.cuh"

namespace adaln {

cudaError_t ln_rows_bf16(const LnArgs &a, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    return rows_vec<DT::BF16>(a, pdl, s, dev);
}

}  // namespace adaln
