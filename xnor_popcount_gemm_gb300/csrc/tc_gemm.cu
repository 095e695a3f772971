// tcgen05 contraction over +1/-1 FP8 / FP4 codes (not built yet).
#include "bt_internal.h"

namespace bt {
bool tc_available() { return false; }
cudaError_t launch_tc_linear(const uint8_t *, const uint8_t *, bt_code, int64_t, int64_t, int64_t, float,
                             void *, bt_dtype, unsigned int *, cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t launch_tc_conv(const uint8_t *, const uint8_t *, bt_code, const ConvGeom &, float, void *,
                           bt_dtype, unsigned int *, cudaStream_t) {
    return cudaErrorNotSupported;
}
}  // namespace bt
