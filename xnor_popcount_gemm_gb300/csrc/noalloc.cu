// bt_binary_linear_noalloc: the binarized linear forward for callers that
// cannot allocate device memory.
//
// bt_binary_linear needs a caller-supplied workspace for the packed
// activations. Some callers cannot obtain one: code that runs inside a host
// framework that owns every device allocation (a plugin's enqueue callback,
// for instance) and code whose memory budget is fixed up front, where a
// cudaMalloc is either not permitted or would stall the device. This entry
// point takes the same inputs and outputs but keeps the packed activations in
// a fixed scratch array compiled into the library, so it allocates nothing.
//
// The array lives in device memory of every GPU that loads the library, from
// load until process exit (kNoallocScratchBytes each). All calls share it:
// two calls whose kernels overlap on the GPU (different streams, or devices
// sharing nothing but a host thread) race on it. Each call's pack kernel
// rewrites every byte it later reads (rows and their zero padding), so
// nothing left by an earlier call needs clearing.
#include "bt_internal.h"

namespace bt {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(16) << 20;   // 16 MiB

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

// In host code `g_noalloc_scratch` names a host-side stand-in, not device
// memory. Its device address is looked up with the caller's device (and
// context) current, once per CUDA context: each context that loads the library
// holds its own copy of the array.
void *scratch_address(cudaError_t *err) {
    static SymbolAddressCache cache;
    return cache.get([](void **p) { return cudaGetSymbolAddress(p, g_noalloc_scratch); }, err);
}

}  // namespace
}  // namespace bt

extern "C" size_t bt_binary_linear_noalloc_max_bytes(void) { return bt::kNoallocScratchBytes; }

extern "C" bt_status bt_binary_linear_noalloc(const void *x, bt_dtype x_dtype, const void *weight, bt_code w_code,
                                              int64_t M, int64_t N, int64_t K, float scale_a, float scale_w,
                                              const float *bias_a, int64_t bias_len, void *out, bt_dtype out_dtype,
                                              bt_algo algo, bt_stream stream) {
    const size_t need = bt_binary_linear_workspace(M, K, x_dtype, w_code);
    if (need > bt::kNoallocScratchBytes) return BT_ERR_WORKSPACE;
    if (need == 0) {
        // nothing to pack (packed x, M == 0, or arguments bt_binary_linear
        // rejects): no scratch, so no address lookup either
        return bt_binary_linear(x, x_dtype, weight, w_code, M, N, K, scale_a, scale_w, bias_a, bias_len, out,
                                out_dtype, algo, nullptr, 0, stream);
    }
    cudaError_t err = cudaSuccess;
    void *scratch = bt::scratch_address(&err);
    if (scratch == nullptr) return BT_ERR_CUDA;
    return bt_binary_linear(x, x_dtype, weight, w_code, M, N, K, scale_a, scale_w, bias_a, bias_len, out,
                            out_dtype, algo, scratch, bt::kNoallocScratchBytes, stream);
}
