// Straight-through backward of the binary linear layer (bitorch-engine
// BinaryLinearForward.backward, whose steps BinaryConv2dForward.backward
// writes out for the convolution):
//   grad_input  = bf16(g @ bf16(sign(w) * scale_w)), zeroed where x / scale_a
//                 (in x's dtype) lies outside [-1, 1]
//   grad_scale_a = sum(grad_input * sign(x) / sqrt(numel(x)))
//   grad_weight = bf16(g^T @ bf16(sign(x) * scale_a))
// Both products run on the tensor cores (tcgen05 kind::f16, bf16 operands,
// fp32 accumulators) through the contraction kernel of tc_gemm.cu. Its
// operands are K-major rows, so the products take:
//   input gradient   A = g [M, N] as is, B = sign(w)^T [K, N] (built once
//                    per weight by bt_sign_transpose); the scale, the rounding
//                    to bf16, the mask and the grad_scale_a terms are fused
//                    into the epilogue;
//   weight gradient  A = g^T [N, M], B = sign(x)^T [K, M], both transposed
//                    here into the workspace.
// sign(v) is torch.sign: (v > 0) - (v < 0), so 0 for zeros and NaN. A +-1 or 0
// operand times a bf16 scale is the page's bf16(sign * scale): the scale is
// rounded to bf16 once on the host and applied to the fp32 sums.
#include <cmath>
#include <type_traits>

#include <cuda_bf16.h>

#include "bt_device.cuh"
#include "bt_internal.h"

namespace bt {
namespace {

constexpr int kTile = 64;           // transpose tile: 64 x 64 elements
constexpr int kTThreads = 256;

__device__ float g_scale_sink;      // grad_scale_a terms when the caller does not want them

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <> __device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }

__device__ __forceinline__ uint16_t sign_bf16(float v) {
    return v > 0.0f ? uint16_t(0x3F80) : (v < 0.0f ? uint16_t(0xBF80) : uint16_t(0));
}

// out[c * ldo + r] = f(in[r * C + c]) for a 64 x 64 tile, through shared
// memory: reads run along c, writes along r, both coalesced. Rows r in
// [R, ldo) are written as 0.
template <typename T, bool SIGN>
__global__ void __launch_bounds__(kTThreads) transpose_kernel(const T *__restrict__ in, int64_t R, int64_t C,
                                                              int64_t ldo, uint16_t *__restrict__ out) {
    __shared__ uint16_t tile[kTile][kTile + 2];
    pdl_launch_dependents();
    pdl_wait();
    in += static_cast<int64_t>(blockIdx.z) * R * C;             // batch of matrices
    out += static_cast<int64_t>(blockIdx.z) * C * ldo;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kTile, c0 = static_cast<int64_t>(blockIdx.x) * kTile;
    for (int i = threadIdx.x; i < kTile * kTile; i += kTThreads) {
        const int rr = i / kTile, cc = i % kTile;
        const int64_t r = r0 + rr, c = c0 + cc;
        uint16_t v = 0;
        if (r < R && c < C) {
            const T x = in[r * C + c];
            if constexpr (SIGN) v = sign_bf16(to_f32<T>(x));
            else v = *reinterpret_cast<const uint16_t *>(&x);
        }
        tile[rr][cc] = v;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kTile * kTile; i += kTThreads) {
        const int cc = i / kTile, rr = i % kTile;
        const int64_t r = r0 + rr, c = c0 + cc;
        if (c < C && r < ldo) out[c * ldo + r] = tile[rr][cc];
    }
}

// torch.sign of two 16-bit values (bf16, or f16 when F16) packed in a word,
// as bf16: 0x3F80 / 0xBF80, 0 for +-0 and NaN (magnitude bits above those of
// infinity).
template <bool F16>
__device__ __forceinline__ uint32_t sign_pair_bf16(uint32_t w) {
    constexpr uint32_t kInf = F16 ? 0x7C00u : 0x7F80u;
    uint32_t r = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t v = (w >> (16 * h)) & 0xFFFFu, mag = v & 0x7FFFu;
        const uint32_t sg = (mag == 0u || mag > kInf) ? 0u : (0x3F80u | (v & 0x8000u));
        r |= sg << (16 * h);
    }
    return r;
}

// Eight consecutive elements of a row as eight bf16 values: torch.sign of
// them (SIGN) or the bf16 values themselves.
template <typename T, bool SIGN>
__device__ __forceinline__ uint4 load8_bf16(const T *p) {
    uint32_t w[4];
    if constexpr (sizeof(T) == 2) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p));
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
        if constexpr (SIGN) {
#pragma unroll
            for (int k = 0; k < 4; ++k) w[k] = sign_pair_bf16<std::is_same<T, __half>::value>(w[k]);
        }
    } else {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
        const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = static_cast<uint32_t>(sign_bf16(f[2 * k])) | (static_cast<uint32_t>(sign_bf16(f[2 * k + 1])) << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Wide form: a 256-thread block moves a 128 x 128 tile through 32 KB of shared
// memory. Loads: every thread takes eight 16-byte chunks (8 elements of a
// row), all in flight at once; 16 threads cover a 256-byte row segment. The
// chunk (row, q) is stored at chunk q ^ (row / 8 mod 16) of its 256-byte
// shared row, so that both the stores here and the 8-row reads below spread
// over all banks. Transpose: each thread reads an 8 x 8 block (8 rows of one
// chunk), pairs rows 2i and 2i+1 column by column with byte permutes, and
// writes output row 2w + p as the words (w, rows 0..7 in pairs) -- 16 bytes
// per output row; 16 threads cover a 256-byte output row segment.
// Needs ldo a multiple of 8. VEC = 16: rows 16-byte aligned (C a multiple of
// 8); VEC = 8: a 2-byte copy whose rows are 8-byte aligned (C a multiple of
// 4), each chunk two 8-byte loads; VEC = 0: element by element. blockIdx.z
// walks a batch of matrices stored one after the other.
template <typename T, bool SIGN, int VEC>
__global__ void __launch_bounds__(kTThreads) transpose8_kernel(const T *__restrict__ in, int64_t R, int64_t C,
                                                               int64_t ldo, uint16_t *__restrict__ out) {
    __shared__ uint4 tile[128 * 16];
    pdl_launch_dependents();
    pdl_wait();
    in += static_cast<int64_t>(blockIdx.z) * R * C;
    out += static_cast<int64_t>(blockIdx.z) * C * ldo;
    const int t = threadIdx.x;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 128, c0 = static_cast<int64_t>(blockIdx.x) * 128;
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int k = i * kTThreads + t, rr = k >> 4, q = k & 15;
        const int64_t r = r0 + rr, c = c0 + 8 * q;
        if constexpr (VEC == 16) {
            v[i] = (r < R && c < C) ? load8_bf16<T, SIGN>(in + r * C + c) : make_uint4(0u, 0u, 0u, 0u);
        } else if constexpr (VEC == 8) {
            static_assert(sizeof(T) == 2 && !SIGN, "8-byte chunks copy 2-byte elements");
            const uint2 lo = (r < R && c < C) ? __ldg(reinterpret_cast<const uint2 *>(in + r * C + c)) : make_uint2(0u, 0u);
            const uint2 hi = (r < R && c + 4 < C) ? __ldg(reinterpret_cast<const uint2 *>(in + r * C + c + 4)) : make_uint2(0u, 0u);
            v[i] = make_uint4(lo.x, lo.y, hi.x, hi.y);
        } else {
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            if (r < R) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if (c + e < C) {
                        const T xv = in[r * C + c + e];
                        uint16_t h;
                        if constexpr (SIGN) h = sign_bf16(to_f32<T>(xv));
                        else h = *reinterpret_cast<const uint16_t *>(&xv);
                        w[e >> 1] |= static_cast<uint32_t>(h) << (16 * (e & 1));
                    }
                }
            }
            v[i] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int k = i * kTThreads + t, rr = k >> 4, q = k & 15;
        tile[rr * 16 + (q ^ ((rr >> 3) & 15))] = v[i];
    }
    __syncthreads();
    const int br = t & 15, bc = t >> 4;
    uint32_t W[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 x = tile[(8 * br + i) * 16 + (bc ^ br)];
        W[i][0] = x.x; W[i][1] = x.y; W[i][2] = x.z; W[i][3] = x.w;
    }
    // rows 2i, 2i+1: X[2i][w] = (M[2i][2w], M[2i+1][2w]), X[2i+1][w] = (.., 2w+1)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t a = W[2 * i][k], b = W[2 * i + 1][k];
            W[2 * i][k] = __byte_perm(a, b, 0x5410);
            W[2 * i + 1][k] = __byte_perm(a, b, 0x7632);
        }
    }
    const int64_t rs = r0 + 8 * br;
    if (rs >= ldo) return;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const int64_t c = c0 + 8 * bc + 2 * w + p;
            if (c < C)
                *reinterpret_cast<uint4 *>(out + c * ldo + rs) = make_uint4(W[p][w], W[2 + p][w], W[4 + p][w], W[6 + p][w]);
        }
    }
}

template <typename T, bool SIGN>
cudaError_t transpose_t(const void *in, int64_t R, int64_t C, int64_t ldo, uint16_t *out, cudaStream_t s,
                        int batch = 1) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute pdl = pdl_attribute();
    cfg.blockDim = dim3(kTThreads);
    cfg.stream = s;
    cfg.attrs = &pdl;
    cfg.numAttrs = 1;
    if (ldo % 8 == 0 && aligned(out, 16) && (ldo + 127) / 128 <= 65535) {
        cfg.gridDim = dim3(static_cast<unsigned>((C + 127) / 128), static_cast<unsigned>((ldo + 127) / 128),
                           static_cast<unsigned>(batch));
        if (C % 8 == 0 && aligned(in, 16))
            return cudaLaunchKernelEx(&cfg, transpose8_kernel<T, SIGN, 16>, static_cast<const T *>(in), R, C, ldo, out);
        if constexpr (sizeof(T) == 2 && !SIGN) {
            if (C % 4 == 0 && aligned(in, 8))
                return cudaLaunchKernelEx(&cfg, transpose8_kernel<T, SIGN, 8>, static_cast<const T *>(in), R, C, ldo, out);
        }
        return cudaLaunchKernelEx(&cfg, transpose8_kernel<T, SIGN, 0>, static_cast<const T *>(in), R, C, ldo, out);
    }
    cfg.gridDim = dim3(static_cast<unsigned>((C + kTile - 1) / kTile), static_cast<unsigned>((ldo + kTile - 1) / kTile),
                       static_cast<unsigned>(batch));
    return cudaLaunchKernelEx(&cfg, transpose_kernel<T, SIGN>, static_cast<const T *>(in), R, C, ldo, out);
}

int64_t round_up64(int64_t v) { return (v + 63) / 64 * 64; }

}  // namespace

cudaError_t launch_transpose_bf16_batched(const void *in, bt_dtype in_t, int64_t R, int64_t C, int64_t ldo, bool sign,
                                          uint16_t *out, int batch, cudaStream_t s) {
    if (R == 0 || C == 0 || batch == 0) return cudaSuccess;
    if (batch < 0 || batch > 65535 || C > (int64_t(65535) * kTile) || ldo > (int64_t(65535) * kTile))
        return cudaErrorInvalidValue;
    if (!sign) return transpose_t<__nv_bfloat16, false>(in, R, C, ldo, out, s, batch);
    switch (in_t) {
        case BT_F32: return transpose_t<float, true>(in, R, C, ldo, out, s, batch);
        case BT_F16: return transpose_t<__half, true>(in, R, C, ldo, out, s, batch);
        default: return transpose_t<__nv_bfloat16, true>(in, R, C, ldo, out, s, batch);
    }
}

cudaError_t launch_transpose_bf16(const void *in, bt_dtype in_t, int64_t R, int64_t C, int64_t ldo, bool sign,
                                  uint16_t *out, cudaStream_t s) {
    if (R == 0 || C == 0) return cudaSuccess;
    if (C > (int64_t(65535) * kTile) || ldo > (int64_t(65535) * kTile)) return cudaErrorInvalidValue;
    if (!sign) return transpose_t<__nv_bfloat16, false>(in, R, C, ldo, out, s);
    switch (in_t) {
        case BT_F32: return transpose_t<float, true>(in, R, C, ldo, out, s);
        case BT_F16: return transpose_t<__half, true>(in, R, C, ldo, out, s);
        default: return transpose_t<__nv_bfloat16, true>(in, R, C, ldo, out, s);
    }
}

}  // namespace bt

using namespace bt;

namespace {
bool finite_pos(float v) { return std::isfinite(v) && v > 0.0f; }
bt_status cuda_status(cudaError_t e) { return e == cudaSuccess ? BT_OK : BT_ERR_CUDA; }
}  // namespace

extern "C" {

int64_t bt_backward_weight_ld(int64_t N) { return N < 0 ? -1 : round_up64(N); }

bt_status bt_sign_transpose(const void *w, bt_dtype w_dtype, int64_t R, int64_t C, int64_t ld, void *out,
                            bt_stream stream) {
    if (w_dtype != BT_F32 && w_dtype != BT_BF16 && w_dtype != BT_F16) return BT_ERR_INVALID_ARG;
    if (R < 0 || C < 0 || ld < R || ld % 8 != 0) return BT_ERR_INVALID_ARG;
    if (C > (int64_t(65535) * 64) || ld > (int64_t(65535) * 64)) return BT_ERR_UNSUPPORTED;
    if (R == 0 || C == 0) return BT_OK;
    if (w == nullptr || out == nullptr) return BT_ERR_INVALID_ARG;
    if (!aligned(w, 16) || !aligned(out, 16)) return BT_ERR_ALIGNMENT;
    return cuda_status(launch_transpose_bf16(w, w_dtype, R, C, ld, true, static_cast<uint16_t *>(out),
                                             reinterpret_cast<cudaStream_t>(stream)));
}

size_t bt_binary_linear_backward_workspace(int64_t M, int64_t N, int64_t K, int want_grad_weight) {
    if (M < 0 || N < 0 || K < 0 || !want_grad_weight) return 0;
    const int64_t ldm = round_up64(M);
    return round_up256(static_cast<size_t>(N * ldm * 2)) + round_up256(static_cast<size_t>(K * ldm * 2));
}

bt_status bt_binary_linear_backward(const void *x, bt_dtype x_dtype, const void *wst, int64_t ldw, const void *g,
                                    int64_t M, int64_t N, int64_t K, float scale_a, float scale_w, void *grad_x,
                                    float *grad_scale_a, void *grad_w, bt_dtype grad_w_dtype, void *workspace,
                                    size_t workspace_bytes, bt_stream stream) {
    if (x_dtype != BT_BF16 && x_dtype != BT_F32) return BT_ERR_INVALID_ARG;
    if (grad_w != nullptr && grad_w_dtype != BT_BF16 && grad_w_dtype != BT_F32) return BT_ERR_INVALID_ARG;
    if (M < 0 || N < 1 || K < 1 || !finite_pos(scale_a) || !finite_pos(scale_w)) return BT_ERR_INVALID_ARG;
    if (N % 8 != 0 || K % 8 != 0) return BT_ERR_UNSUPPORTED;
    if (M > (int64_t(1) << 30) || N > (int64_t(1) << 30) || K > (int64_t(1) << 30)) return BT_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (M == 0) {
        // empty batch (grad_x is empty too): the sum is zero, grad_w = 0
        if (grad_scale_a != nullptr && cudaMemsetAsync(grad_scale_a, 0, sizeof(float), s) != cudaSuccess) return BT_ERR_CUDA;
        if (grad_w != nullptr &&
            cudaMemsetAsync(grad_w, 0, static_cast<size_t>(N * K) * (grad_w_dtype == BT_F32 ? 4 : 2), s) != cudaSuccess)
            return BT_ERR_CUDA;
        return BT_OK;
    }
    if (grad_scale_a != nullptr && grad_x == nullptr) return BT_ERR_INVALID_ARG;
    if (grad_x != nullptr && (wst == nullptr || ldw < N || ldw % 8 != 0)) return BT_ERR_INVALID_ARG;
    if (x == nullptr || g == nullptr) return BT_ERR_INVALID_ARG;
    if (!tc_available()) return BT_ERR_UNSUPPORTED;
    if (!aligned(x, 16) || !aligned(g, 16) || (wst && !aligned(wst, 16)) || (grad_x && !aligned(grad_x, 16)) ||
        (grad_w && !aligned(grad_w, 16)) || (grad_scale_a && !aligned(grad_scale_a, 4)))
        return BT_ERR_ALIGNMENT;
    const size_t need = bt_binary_linear_backward_workspace(M, N, K, grad_w != nullptr);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return BT_ERR_WORKSPACE;
    if (need > 0 && !aligned(workspace, 256)) return BT_ERR_ALIGNMENT;
    unsigned int *err = device_error_word();
    if (err == nullptr) return BT_ERR_CUDA;

    if (grad_x != nullptr) {
        float *sum = grad_scale_a;
        if (sum == nullptr) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_scale_sink) != cudaSuccess) return BT_ERR_CUDA;
            sum = static_cast<float *>(p);
        }
        if (cudaMemsetAsync(sum, 0, sizeof(float), s) != cudaSuccess) return BT_ERR_CUDA;
        TcMask mk{x, x_dtype, scale_a, static_cast<float>(1.0 / std::sqrt(static_cast<double>(M) * static_cast<double>(K))),
                  sum};
        const cudaError_t e = launch_tc_bf16(static_cast<const uint16_t *>(g), N, static_cast<const uint16_t *>(wst), ldw,
                                             M, K, N, bf16_round_host(scale_w), grad_x, BT_BF16, &mk, err, s);
        if (e != cudaSuccess) return BT_ERR_CUDA;
    }
    if (grad_w != nullptr) {
        const int64_t ldm = round_up64(M);
        uint16_t *gt = static_cast<uint16_t *>(workspace);
        uint16_t *xst = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(workspace) +
                                                     round_up256(static_cast<size_t>(N * ldm * 2)));
        if (launch_transpose_bf16(g, BT_BF16, M, N, ldm, false, gt, s) != cudaSuccess ||
            launch_transpose_bf16(x, x_dtype, M, K, ldm, true, xst, s) != cudaSuccess)
            return BT_ERR_CUDA;
        // the contraction runs over the zero-padded length ldm: the pads add 0
        const cudaError_t e = launch_tc_bf16(gt, ldm, xst, ldm, N, K, ldm, bf16_round_host(scale_a), grad_w,
                                             grad_w_dtype, nullptr, err, s);
        if (e != cudaSuccess) return BT_ERR_CUDA;
    }
    return BT_OK;
}

}  // extern "C"
