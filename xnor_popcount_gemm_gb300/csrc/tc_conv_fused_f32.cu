// The implicit-im2col binary convolution that packs its own input, for x of
// f32: the instantiations of one input type (the kernel lives in
// tc_conv_kernel.cuh).
#include "tc_conv_kernel.cuh"

namespace bt {
namespace conv {

cudaError_t launch_fused_f32(const CUtensorMap &ma, const ConvPlan &p, bt_code code, bt_dtype out_t, cudaStream_t s) {
    return launch_code<float>(ma, ma, p, code, out_t, s);
}

}  // namespace conv
}  // namespace bt
