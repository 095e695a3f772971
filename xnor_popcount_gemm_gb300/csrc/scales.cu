// Activation scale on the device (bitorch-engine BinaryConv2dCutlass.set_activation):
// on the first forward, scale_a = (2 * x.abs().mean()) for a symmetric layer or
// (4 * x.abs().mean()) otherwise, stored in the layer's dtype. Computed here
// without a host round trip: the sum of |x| in double (exact for bf16 and f16
// inputs of any realistic range; one rounding per block sum for f32), the mean
// rounded once to x's dtype (x.abs().mean() is a tensor of x's dtype), times
// the factor, rounded to the layer's dtype, written as one float that
// bt_binary_linear_dscale / bt_binary_conv2d_dscale read.
#include <cmath>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bt_device.cuh"
#include "bt_internal.h"

namespace bt {
namespace {

constexpr int kThreads = 256;

template <typename T> __device__ __forceinline__ double abs_d(T v);
template <> __device__ __forceinline__ double abs_d<float>(float v) { return fabs(static_cast<double>(v)); }
template <> __device__ __forceinline__ double abs_d<__nv_bfloat16>(__nv_bfloat16 v) {
    return fabs(static_cast<double>(__bfloat162float(v)));
}
template <> __device__ __forceinline__ double abs_d<__half>(__half v) { return fabs(static_cast<double>(__half2float(v))); }

template <typename T>
__global__ void __launch_bounds__(kThreads) abs_sum_kernel(const T *__restrict__ x, int64_t n, double *__restrict__ acc) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ double part[kThreads / 32];
    double v = 0.0;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * kThreads)
        v += abs_d<T>(x[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < kThreads / 32; ++w) t += part[w];
        atomicAdd(acc, t);
    }
}

// Round a double to the nearest value with `bits` significand bits (ties to
// even), within the normal range of the target type.
__device__ __forceinline__ double round_sig(double v, int bits) {
    unsigned long long u = static_cast<unsigned long long>(__double_as_longlong(v));
    const int drop = 52 - (bits - 1);
    const unsigned long long half = (1ull << (drop - 1)) - 1ull + ((u >> drop) & 1ull);
    u = (u + half) & ~((1ull << drop) - 1ull);
    return __longlong_as_double(static_cast<long long>(u));
}

// v rounded to dtype t (bf16: 8 significand bits, f16: 11, f32: 24), as a float.
__device__ __forceinline__ float round_to(double v, int t) {
    if (t == BT_BF16) {
        if (fabs(v) < 1.1754943508222875e-38) return __bfloat162float(__float2bfloat16_rn(__double2float_rn(v)));
        const double r = round_sig(v, 8);
        return fabs(r) > 3.3895313892515355e38 ? (r > 0 ? INFINITY : -INFINITY) : static_cast<float>(r);
    }
    if (t == BT_F16) {
        if (fabs(v) < 6.103515625e-05) return __half2float(__float2half_rn(__double2float_rn(v)));
        const double r = round_sig(v, 11);
        return fabs(r) > 65504.0 ? (r > 0 ? INFINITY : -INFINITY) : static_cast<float>(r);
    }
    return __double2float_rn(v);
}

__global__ void finish_kernel(const double *__restrict__ acc, int64_t n, float factor, int x_t, int scale_t,
                              float *__restrict__ out) {
    pdl_launch_dependents();
    pdl_wait();
    const float mean = round_to(*acc / static_cast<double>(n), x_t);                    // x.abs().mean()
    const float scaled = round_to(static_cast<double>(factor) * static_cast<double>(mean), x_t);   // factor * mean
    *out = round_to(static_cast<double>(scaled), scale_t);                              // .to(layer dtype)
}

__device__ double g_abs_sum[128];
__device__ double g_abs_sum_fused;

}  // namespace

// Accumulator of the forwards that initialise scale_a while they pack x (one
// per CUDA context), as seen from the current context.
double *fused_abs_sum_accumulator(cudaError_t *err) {
    static SymbolAddressCache cache;
    return static_cast<double *>(cache.get([](void **p) { return cudaGetSymbolAddress(p, g_abs_sum_fused); }, err));
}

cudaError_t launch_abs_sum(const void *x, bt_dtype x_dtype, int64_t n, double *acc, cudaStream_t s) {
    int64_t blocks = (n + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    switch (x_dtype) {
        case BT_F32:
            return launch_pdl(abs_sum_kernel<float>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), s,
                              static_cast<const float *>(x), n, acc);
        case BT_F16:
            return launch_pdl(abs_sum_kernel<__half>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), s,
                              static_cast<const __half *>(x), n, acc);
        default:
            return launch_pdl(abs_sum_kernel<__nv_bfloat16>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), s,
                              static_cast<const __nv_bfloat16 *>(x), n, acc);
    }
}

cudaError_t launch_scale_finish(const double *acc, int64_t n, float factor, bt_dtype x_dtype, bt_dtype scale_dtype,
                                float *scale_out, cudaStream_t s) {
    return launch_pdl(finish_kernel, dim3(1), dim3(1), s, acc, n, factor, static_cast<int>(x_dtype),
                      static_cast<int>(scale_dtype), scale_out);
}

}  // namespace bt

using namespace bt;

extern "C" {

bt_status bt_scale_init(const void *x, bt_dtype x_dtype, int64_t n, float factor, bt_dtype scale_dtype,
                        float *scale_out, bt_stream stream) {
    if (x_dtype != BT_F32 && x_dtype != BT_BF16 && x_dtype != BT_F16) return BT_ERR_INVALID_ARG;
    if (scale_dtype != BT_F32 && scale_dtype != BT_BF16 && scale_dtype != BT_F16) return BT_ERR_INVALID_ARG;
    if (n < 1 || !(std::isfinite(factor) && factor > 0.0f)) return BT_ERR_INVALID_ARG;
    if (x == nullptr || scale_out == nullptr) return BT_ERR_INVALID_ARG;
    if (!aligned(x, static_cast<size_t>(dtype_bytes(x_dtype))) || !aligned(scale_out, 4)) return BT_ERR_ALIGNMENT;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return BT_ERR_CUDA;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_abs_sum) != cudaSuccess) return BT_ERR_CUDA;
    // one accumulator per device; calls on one device run in stream order
    double *acc = static_cast<double *>(p) + dev;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(acc, 0, sizeof(double), s) != cudaSuccess) return BT_ERR_CUDA;
    int64_t blocks = (n + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    cudaError_t e;
    switch (x_dtype) {
        case BT_F32:
            e = launch_pdl(abs_sum_kernel<float>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), s,
                           static_cast<const float *>(x), n, acc);
            break;
        case BT_F16:
            e = launch_pdl(abs_sum_kernel<__half>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), s,
                           static_cast<const __half *>(x), n, acc);
            break;
        default:
            e = launch_pdl(abs_sum_kernel<__nv_bfloat16>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), s,
                           static_cast<const __nv_bfloat16 *>(x), n, acc);
            break;
    }
    if (e != cudaSuccess) return BT_ERR_CUDA;
    e = launch_pdl(finish_kernel, dim3(1), dim3(1), s, static_cast<const double *>(acc), n, factor,
                   static_cast<int>(x_dtype), static_cast<int>(scale_dtype), scale_out);
    return e == cudaSuccess ? BT_OK : BT_ERR_CUDA;
}

}  // extern "C"
