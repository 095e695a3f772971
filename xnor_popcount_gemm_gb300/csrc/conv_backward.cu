// Straight-through backward of the binary conv2d layer (bitorch-engine
// BinaryConv2dForward.backward):
//   wt           = bf16(sign(w) * scale_w)
//   grad_input   = conv2d_input(x.shape, wt, g), rounded to bf16, times the
//                  mask middle = !(q < -1 || q > 1), q = x / scale_a in x's dtype
//   grad_scale_a = sum(grad_input * sign(x) / sqrt(numel(x)))
//   grad_weight  = conv2d_weight(bf16(sign(x) * scale_a), w.shape, g)
// Both gradients are lowered to matrix products on the tensor cores (bf16
// operands, fp32 accumulators; tc_gemm.cu), the unfold + mm reading of a
// convolution run backwards. With P = B*Ho*Wo output pixels and taps
// t = (c, kh, kw) (OIHW order, C*k*k of them):
//   input gradient   D[t, p] = bf16(scale_w) * sum_o sign(w)[o, t] * g[p, o]
//                    (A = sign(w)^T [t, O] from bt_sign_transpose, B = g per
//                    pixel [P, O], transposed image by image); then each input
//                    element gathers the D entries of the taps that read it
//                    (col2im, fp32), rounds once to bf16, and takes the mask
//                    and its grad_scale_a term.
//   weight gradient  grad_w[o, t] = bf16(scale_a) * sum_p g[o, p] * sign(x)[p, t]
//                    (A = g as [O, P] rows, B = the im2col of sign(x)
//                    transposed [t, P], zeros for taps in the padding); the
//                    long sum over P is split in K, the parts added in fp32.
#include <cmath>
#include <cstring>

#include <cuda_bf16.h>

#include "bt_device.cuh"
#include "bt_internal.h"

namespace bt {
namespace {

constexpr int kThreads = 256;

struct ConvBwdGeom {
    int64_t B, C, H, W, O, Ho, Wo, P, T;   // T = C*k*k taps
    int k, s, p, d;
};

__device__ __forceinline__ uint16_t sign_bf16_f(float v) {
    return v > 0.0f ? uint16_t(0x3F80) : (v < 0.0f ? uint16_t(0xBF80) : uint16_t(0));
}

template <typename T> __device__ __forceinline__ float ld_f32(const T *p, int64_t i);
template <> __device__ __forceinline__ float ld_f32<float>(const float *p, int64_t i) { return __ldg(p + i); }
template <> __device__ __forceinline__ float ld_f32<__nv_bfloat16>(const __nv_bfloat16 *p, int64_t i) {
    return __bfloat162float(p[i]);
}

// g [B, O, Ho*Wo] -> go [O, ldp]: row o holds g[b, o, :] for b = 0, 1, ...
// one after the other; columns P .. ldp-1 are 0.
__global__ void __launch_bounds__(kThreads) g_rows_kernel(const uint16_t *__restrict__ g, ConvBwdGeom q, int64_t ldp,
                                                          uint16_t *__restrict__ go) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t hw = q.Ho * q.Wo, total = q.O * ldp;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * kThreads) {
        const int64_t o = i / ldp, col = i - o * ldp;
        uint16_t v = 0;
        if (col < q.P) {
            const int64_t b = col / hw, pix = col - b * hw;
            v = g[(b * q.O + o) * hw + pix];
        }
        go[i] = v;
    }
}

// im2col of sign(x), transposed: u[t, p] (row pitch ldp) = sign(x[b, c, ih, iw])
// as bf16 for tap t = (c, kh, kw) of output pixel p = (b, i, j), ih = i*s - p
// + kh*d, iw = j*s - p + kw*d; 0 in the padding and for p >= P.
template <typename T>
__global__ void __launch_bounds__(kThreads) sign_im2col_t_kernel(const T *__restrict__ x, ConvBwdGeom q, int64_t ldp,
                                                                 uint16_t *__restrict__ u) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t total = q.T * ldp, hw = q.Ho * q.Wo, kk = static_cast<int64_t>(q.k) * q.k;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * kThreads) {
        const int64_t t = i / ldp, col = i - t * ldp;
        uint16_t v = 0;
        if (col < q.P) {
            const int64_t c = t / kk, tap = t - c * kk;
            const int kh = static_cast<int>(tap / q.k), kw = static_cast<int>(tap - static_cast<int64_t>(kh) * q.k);
            const int64_t b = col / hw, pix = col - b * hw;
            const int64_t oi = pix / q.Wo, oj = pix - oi * q.Wo;
            const int64_t ih = oi * q.s - q.p + static_cast<int64_t>(kh) * q.d;
            const int64_t iw = oj * q.s - q.p + static_cast<int64_t>(kw) * q.d;
            if (ih >= 0 && ih < q.H && iw >= 0 && iw < q.W) v = sign_bf16_f(ld_f32<T>(x, ((b * q.C + c) * q.H + ih) * q.W + iw));
        }
        u[i] = v;
    }
}

// col2im of D [T, P] (fp32, row pitch P) into the input gradient, with the
// straight-through mask and the grad_scale_a terms: one thread per input
// element (b, c, h, w), w fastest. Taps are summed in (kh, kw) order.
template <typename T>
__global__ void __launch_bounds__(kThreads) col2im_mask_kernel(const float *__restrict__ dt, const T *__restrict__ x,
                                                               ConvBwdGeom q, float scale_a, float norm,
                                                               __nv_bfloat16 *__restrict__ gx, float *__restrict__ sum) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t total = q.B * q.C * q.H * q.W;
    float tsum = 0.0f;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * kThreads) {
        const int64_t w = e % q.W, r1 = e / q.W, h = r1 % q.H, r2 = r1 / q.H, c = r2 % q.C, b = r2 / q.C;
        float acc = 0.0f;
        for (int kh = 0; kh < q.k; ++kh) {
            const int64_t hn = h + q.p - static_cast<int64_t>(kh) * q.d;
            if (hn < 0 || hn % q.s != 0 || hn / q.s >= q.Ho) continue;
            const int64_t i = hn / q.s;
            for (int kw = 0; kw < q.k; ++kw) {
                const int64_t wn = w + q.p - static_cast<int64_t>(kw) * q.d;
                if (wn < 0 || wn % q.s != 0 || wn / q.s >= q.Wo) continue;
                const int64_t j = wn / q.s;
                const int64_t t = (c * q.k + kh) * q.k + kw;
                acc = __fadd_rn(acc, __ldg(dt + t * q.P + (b * q.Ho + i) * q.Wo + j));
            }
        }
        const float y = __bfloat162float(__float2bfloat16_rn(acc));
        const float xv = ld_f32<T>(x, e);
        float qv = __fdiv_rn(xv, scale_a);
        if constexpr (sizeof(T) == 2) qv = __bfloat162float(__float2bfloat16_rn(qv));
        const float ym = __fmul_rn(y, (qv < -1.0f || qv > 1.0f) ? 0.0f : 1.0f);
        const float sg = (xv > 0.0f ? 1.0f : 0.0f) - (xv < 0.0f ? 1.0f : 0.0f);
        tsum = __fadd_rn(tsum, __fmul_rn(__fmul_rn(ym, sg), norm));
        gx[e] = __float2bfloat16_rn(ym);                      // ym is bf16-exact
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tsum += __shfl_xor_sync(0xFFFFFFFFu, tsum, o);
    if ((threadIdx.x & 31) == 0) atomicAdd(sum, tsum);
}

// grad_w[i] = out_t(alpha * sum over the K splits of part[s][i]), fp32 sums in
// split order.
template <typename O>
__global__ void __launch_bounds__(kThreads) split_sum_kernel(const float *__restrict__ part, int splits, int64_t n,
                                                             float alpha, O *__restrict__ out) {
    pdl_launch_dependents();
    pdl_wait();
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * kThreads) {
        float acc = 0.0f;
        for (int sp = 0; sp < splits; ++sp) acc = __fadd_rn(acc, __ldg(part + sp * n + i));
        const float v = __fmul_rn(acc, alpha);
        if constexpr (sizeof(O) == 4) out[i] = v;
        else out[i] = __float2bfloat16_rn(v);
    }
}

template <typename K, typename... Args>
cudaError_t launch_flat(K kern, int64_t work, cudaStream_t s, Args... args) {
    int64_t blocks = (work + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute pdl = pdl_attribute();
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cfg.attrs = &pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

float bf16_round_h(float v) {
    uint32_t u;
    std::memcpy(&u, &v, 4);
    if ((u & 0x7F800000u) == 0x7F800000u) return v;
    u = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
    float r;
    std::memcpy(&r, &u, 4);
    return r;
}

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

// Pieces of the workspace. The input gradient's (g per pixel, D) and the
// weight gradient's (g rows, sign(x) im2col, partial sums) run one after the
// other on the stream, so they share the space.
struct ConvBwdPlan {
    ConvBwdGeom q;
    int splits;
    int64_t ldp;          // padded P of the weight gradient's rows
    size_t gp_off, dt_off, dgrad_bytes;
    size_t go_off, u_off, part_off, wgrad_bytes;
};

bool make_plan(int64_t B, int64_t C, int64_t H, int64_t W, int64_t O, int k, int s, int p, int d, ConvBwdPlan &pl) {
    ConvBwdGeom &q = pl.q;
    q.B = B; q.C = C; q.H = H; q.W = W; q.O = O; q.k = k; q.s = s; q.p = p; q.d = d;
    const int64_t hn = H + 2 * static_cast<int64_t>(p) - static_cast<int64_t>(d) * (k - 1) - 1;
    const int64_t wn = W + 2 * static_cast<int64_t>(p) - static_cast<int64_t>(d) * (k - 1) - 1;
    if (hn < 0 || wn < 0) return false;
    q.Ho = hn / s + 1;
    q.Wo = wn / s + 1;
    q.P = B * q.Ho * q.Wo;
    q.T = C * k * k;
    // K splits for the weight gradient: about two units of work per CTA pair
    const int64_t tiles = ((O + 255) / 256) * ((q.T + 223) / 224);
    int64_t sp = (76 + tiles - 1) / tiles;
    if (sp > 64) sp = 64;
    if (sp < 1) sp = 1;
    while (sp > 1 && q.P / sp < 512) --sp;                   // keep >= 8 slices per split
    pl.splits = static_cast<int>(sp);
    pl.ldp = (q.P + 64 * sp - 1) / (64 * sp) * (64 * sp);
    pl.gp_off = 0;
    pl.dt_off = up256(static_cast<size_t>(q.P * O * 2));
    pl.dgrad_bytes = pl.dt_off + up256(static_cast<size_t>(q.T * q.P * 4));
    pl.go_off = 0;
    pl.u_off = up256(static_cast<size_t>(O * pl.ldp * 2));
    pl.part_off = pl.u_off + up256(static_cast<size_t>(q.T * pl.ldp * 2));
    pl.wgrad_bytes = pl.part_off + up256(static_cast<size_t>(sp * O * q.T * 4));
    return true;
}

__device__ float g_conv_scale_sink;

}  // namespace
}  // namespace bt

using namespace bt;

extern "C" {

size_t bt_binary_conv2d_backward_workspace(int64_t B, int64_t C, int64_t H, int64_t W, int64_t O, int kernel_size,
                                           int stride, int padding, int dilation, int want_grad_input,
                                           int want_grad_weight) {
    ConvBwdPlan pl;
    if (B < 0 || C < 1 || H < 1 || W < 1 || O < 1 || kernel_size < 1 || stride < 1 || padding < 0 || dilation < 1 ||
        !make_plan(B, C, H, W, O, kernel_size, stride, padding, dilation, pl))
        return 0;
    size_t need = 0;
    if (want_grad_input && pl.dgrad_bytes > need) need = pl.dgrad_bytes;
    if (want_grad_weight && pl.wgrad_bytes > need) need = pl.wgrad_bytes;
    return need;
}

bt_status bt_binary_conv2d_backward(const void *x, bt_dtype x_dtype, const void *wst, int64_t ldw, const void *g,
                                    int64_t B, int64_t C, int64_t H, int64_t W, int64_t O, int kernel_size, int stride,
                                    int padding, int dilation, float scale_a, float scale_w, void *grad_x,
                                    float *grad_scale_a, void *grad_w, bt_dtype grad_w_dtype, void *workspace,
                                    size_t workspace_bytes, bt_stream stream) {
    if (x_dtype != BT_BF16 && x_dtype != BT_F32) return BT_ERR_INVALID_ARG;
    if (grad_w != nullptr && grad_w_dtype != BT_BF16 && grad_w_dtype != BT_F32) return BT_ERR_INVALID_ARG;
    if (B < 0 || C < 1 || H < 1 || W < 1 || O < 1 || kernel_size < 1 || stride < 1 || padding < 0 || dilation < 1)
        return BT_ERR_INVALID_ARG;
    if (!(std::isfinite(scale_a) && scale_a > 0.0f && std::isfinite(scale_w) && scale_w > 0.0f)) return BT_ERR_INVALID_ARG;
    if (H > (1 << 20) || W > (1 << 20) || kernel_size > 64 || padding > (1 << 20) || stride > (1 << 20) ||
        dilation > (1 << 10) || C > (int64_t(1) << 24) || O > (int64_t(1) << 24))
        return BT_ERR_UNSUPPORTED;
    ConvBwdPlan pl;
    if (!make_plan(B, C, H, W, O, kernel_size, stride, padding, dilation, pl)) return BT_ERR_INVALID_ARG;
    const ConvBwdGeom &q = pl.q;
    if (O % 8 != 0 || B > 65535) return BT_ERR_UNSUPPORTED;
    if (q.P > (int64_t(1) << 31) - 512 || q.T > (int64_t(1) << 24)) return BT_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (B == 0) {
        if (grad_scale_a != nullptr && cudaMemsetAsync(grad_scale_a, 0, sizeof(float), s) != cudaSuccess) return BT_ERR_CUDA;
        if (grad_w != nullptr &&
            cudaMemsetAsync(grad_w, 0, static_cast<size_t>(O * q.T) * (grad_w_dtype == BT_F32 ? 4 : 2), s) != cudaSuccess)
            return BT_ERR_CUDA;
        return BT_OK;
    }
    if (grad_scale_a != nullptr && grad_x == nullptr) return BT_ERR_INVALID_ARG;
    if (grad_x != nullptr && (wst == nullptr || ldw < O || ldw % 8 != 0)) return BT_ERR_INVALID_ARG;
    if (x == nullptr || g == nullptr) return BT_ERR_INVALID_ARG;
    if (!tc_available()) return BT_ERR_UNSUPPORTED;
    if (!aligned(x, 16) || !aligned(g, 16) || (wst && !aligned(wst, 16)) || (grad_x && !aligned(grad_x, 16)) ||
        (grad_w && !aligned(grad_w, 16)) || (grad_scale_a && !aligned(grad_scale_a, 4)))
        return BT_ERR_ALIGNMENT;
    const size_t need = bt_binary_conv2d_backward_workspace(B, C, H, W, O, kernel_size, stride, padding, dilation,
                                                            grad_x != nullptr, grad_w != nullptr);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return BT_ERR_WORKSPACE;
    if (need > 0 && !aligned(workspace, 256)) return BT_ERR_ALIGNMENT;
    unsigned int *err = device_error_word();
    if (err == nullptr) return BT_ERR_CUDA;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const uint16_t *g16 = static_cast<const uint16_t *>(g);

    if (grad_x != nullptr) {
        float *sum = grad_scale_a;
        if (sum == nullptr) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_conv_scale_sink) != cudaSuccess) return BT_ERR_CUDA;
            sum = static_cast<float *>(p);
        }
        uint16_t *gp = reinterpret_cast<uint16_t *>(ws + pl.gp_off);
        float *dt = reinterpret_cast<float *>(ws + pl.dt_off);
        // g per pixel: [B] x ([O, Ho*Wo] -> [Ho*Wo, O])
        if (cudaMemsetAsync(sum, 0, sizeof(float), s) != cudaSuccess ||
            launch_transpose_bf16_batched(g16, BT_BF16, O, q.Ho * q.Wo, O, false, gp, static_cast<int>(B), s) !=
                cudaSuccess)
            return BT_ERR_CUDA;
        if (launch_tc_bf16(static_cast<const uint16_t *>(wst), ldw, gp, O, q.T, q.P, O, bf16_round_h(scale_w), dt, BT_F32,
                           nullptr, err, s) != cudaSuccess)
            return BT_ERR_CUDA;
        const float norm = static_cast<float>(1.0 / std::sqrt(static_cast<double>(B) * C * H * W));
        const int64_t n = B * C * H * W;
        const cudaError_t e =
            x_dtype == BT_F32
                ? launch_flat(col2im_mask_kernel<float>, n, s, dt, static_cast<const float *>(x), q, scale_a, norm,
                              static_cast<__nv_bfloat16 *>(grad_x), sum)
                : launch_flat(col2im_mask_kernel<__nv_bfloat16>, n, s, dt, static_cast<const __nv_bfloat16 *>(x), q,
                              scale_a, norm, static_cast<__nv_bfloat16 *>(grad_x), sum);
        if (e != cudaSuccess) return BT_ERR_CUDA;
    }
    if (grad_w != nullptr) {
        uint16_t *go = reinterpret_cast<uint16_t *>(ws + pl.go_off);
        uint16_t *u = reinterpret_cast<uint16_t *>(ws + pl.u_off);
        float *part = reinterpret_cast<float *>(ws + pl.part_off);
        cudaError_t e = launch_flat(g_rows_kernel, q.O * pl.ldp, s, g16, q, pl.ldp, go);
        if (e == cudaSuccess)
            e = x_dtype == BT_F32
                    ? launch_flat(sign_im2col_t_kernel<float>, q.T * pl.ldp, s, static_cast<const float *>(x), q, pl.ldp, u)
                    : launch_flat(sign_im2col_t_kernel<__nv_bfloat16>, q.T * pl.ldp, s,
                                  static_cast<const __nv_bfloat16 *>(x), q, pl.ldp, u);
        if (e == cudaSuccess) e = launch_tc_bf16_splitk(go, pl.ldp, u, pl.ldp, O, q.T, pl.ldp, pl.splits, 1.0f, part, err, s);
        if (e == cudaSuccess)
            e = grad_w_dtype == BT_F32
                    ? launch_flat(split_sum_kernel<float>, O * q.T, s, static_cast<const float *>(part), pl.splits, O * q.T,
                                  bf16_round_h(scale_a), static_cast<float *>(grad_w))
                    : launch_flat(split_sum_kernel<__nv_bfloat16>, O * q.T, s, static_cast<const float *>(part), pl.splits,
                                  O * q.T, bf16_round_h(scale_a), static_cast<__nv_bfloat16 *>(grad_w));
        if (e != cudaSuccess) return BT_ERR_CUDA;
    }
    return BT_OK;
}

}  // extern "C"
