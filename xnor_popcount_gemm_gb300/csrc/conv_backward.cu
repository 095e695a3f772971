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

// The kernels below map rows to blockIdx.y (looping when there are more
// rows than grid rows) and the elements of a row to threads, so that every
// index is a 32-bit quotient of a row position; sizes are validated to fit.

// g [B, O, Ho*Wo] -> go [O, ldp]: row o holds g[b, o, :] for b = 0, 1, ...
// one after the other; columns P .. ldp-1 are 0. A thread copies its column
// of kGRows rows, all the loads issued before the stores.
constexpr int kGRows = 8;
__global__ void __launch_bounds__(kThreads) g_rows_kernel(const uint16_t *__restrict__ g, ConvBwdGeom q, int64_t ldp,
                                                          uint16_t *__restrict__ go) {
    pdl_launch_dependents();
    pdl_wait();
    const uint32_t hw = static_cast<uint32_t>(q.Ho * q.Wo);
    const uint32_t col = blockIdx.x * kThreads + threadIdx.x;
    if (col >= ldp) return;
    const bool live = col < q.P;
    const uint32_t b = live ? col / hw : 0u, pix = col - b * hw;
    const uint16_t *src = g + static_cast<int64_t>(b) * q.O * hw + pix;
    for (int64_t o0 = static_cast<int64_t>(blockIdx.y) * kGRows; o0 < q.O; o0 += static_cast<int64_t>(gridDim.y) * kGRows) {
        uint16_t v[kGRows];
#pragma unroll
        for (int r = 0; r < kGRows; ++r) v[r] = (live && o0 + r < q.O) ? src[(o0 + r) * hw] : uint16_t(0);
#pragma unroll
        for (int r = 0; r < kGRows; ++r)
            if (o0 + r < q.O) go[(o0 + r) * ldp + col] = v[r];
    }
}

// The same, four columns per thread as one 8-byte copy, where an image's
// Ho*Wo pixels are a multiple of 4 (each group of four columns then lies in
// one image, and its source and destination are 8-byte aligned).
__global__ void __launch_bounds__(kThreads) g_rows4_kernel(const uint16_t *__restrict__ g, ConvBwdGeom q, int64_t ldp,
                                                           uint16_t *__restrict__ go) {
    pdl_launch_dependents();
    pdl_wait();
    const uint32_t hw = static_cast<uint32_t>(q.Ho * q.Wo);
    const uint32_t col = 4u * (blockIdx.x * kThreads + threadIdx.x);
    if (col >= ldp) return;
    const bool live = col < q.P;
    const uint32_t b = live ? col / hw : 0u, pix = col - b * hw;
    const uint16_t *src = g + static_cast<int64_t>(b) * q.O * hw + pix;
    for (int64_t o0 = static_cast<int64_t>(blockIdx.y) * kGRows; o0 < q.O; o0 += static_cast<int64_t>(gridDim.y) * kGRows) {
        uint2 v[kGRows];
#pragma unroll
        for (int r = 0; r < kGRows; ++r)
            v[r] = (live && o0 + r < q.O) ? __ldg(reinterpret_cast<const uint2 *>(src + (o0 + r) * hw)) : make_uint2(0u, 0u);
#pragma unroll
        for (int r = 0; r < kGRows; ++r)
            if (o0 + r < q.O) *reinterpret_cast<uint2 *>(go + (o0 + r) * ldp + col) = v[r];
    }
}

// im2col of sign(x), transposed: u[t, p] (row pitch ldp) = sign(x[b, c, ih, iw])
// as bf16 for tap t = (c, kh, kw) of output pixel p = (b, i, j), ih = i*s - p
// + kh*d, iw = j*s - p + kw*d; 0 in the padding and for p >= P. A thread
// keeps its pixel p and walks kTapRows consecutive taps, stepping (c, kh, kw),
// (ih, iw), its channel plane and its output row without divisions or 64-bit
// products (offsets within a plane are below H*W < 2^31).
constexpr int kTapRows = 16;
template <typename T>
__global__ void __launch_bounds__(kThreads) sign_im2col_t_kernel(const T *__restrict__ x, ConvBwdGeom q, int64_t ldp,
                                                                 uint16_t *__restrict__ u) {
    pdl_launch_dependents();
    pdl_wait();
    const uint32_t col = blockIdx.x * kThreads + threadIdx.x;
    if (col >= ldp) return;
    const uint32_t hw = static_cast<uint32_t>(q.Ho * q.Wo), wo = static_cast<uint32_t>(q.Wo);
    const bool live = col < q.P;
    const uint32_t b = live ? col / hw : 0u, pix = col - b * hw, oi = pix / wo, oj = pix - oi * wo;
    const int h0 = static_cast<int>(oi) * q.s - q.p, w0 = static_cast<int>(oj) * q.s - q.p;
    const int H = static_cast<int>(q.H), W = static_cast<int>(q.W), k = q.k, d = q.d;
    const int64_t HW = q.H * q.W;
    const T *xb = x + static_cast<int64_t>(b) * q.C * HW;
    const uint32_t kk = static_cast<uint32_t>(k * k);
    for (int64_t t0 = static_cast<int64_t>(blockIdx.y) * kTapRows; t0 < q.T;
         t0 += static_cast<int64_t>(gridDim.y) * kTapRows) {
        const uint32_t c = static_cast<uint32_t>(t0) / kk, tap = static_cast<uint32_t>(t0) - c * kk;
        int kh = static_cast<int>(tap) / k, kw = static_cast<int>(tap) - kh * k;
        int ih = h0 + kh * d, iw = w0 + kw * d;
        const T *xc = xb + static_cast<int64_t>(c) * HW;
        uint16_t *ur = u + t0 * ldp + col;
        const int n = static_cast<int>(t0 + kTapRows < q.T ? kTapRows : q.T - t0);
        for (int i = 0; i < n; ++i, ur += ldp) {
            uint16_t v = 0;
            if (live && static_cast<unsigned>(ih) < static_cast<unsigned>(H) && static_cast<unsigned>(iw) < static_cast<unsigned>(W))
                v = sign_bf16_f(ld_f32<T>(xc, ih * W + iw));
            *ur = v;
            iw += d;
            if (++kw == k) {
                kw = 0;
                iw = w0;
                ih += d;
                if (++kh == k) {
                    kh = 0;
                    ih = h0;
                    xc += HW;
                }
            }
        }
    }
}

// col2im of D [T, P] (fp32, row pitch P) into the input gradient, with the
// straight-through mask and the grad_scale_a terms: one thread per input
// element (b, c, h, w) of an image plane (b, c) (blockIdx.y), w fastest.
// The taps that read (h, w) -- kh with h + p - kh*d = i*s, 0 <= i < Ho, and
// the same for w -- are listed once per thread (S = the stride when it is 1
// or 2, so the divisions become shifts; 0 for any stride); taps are summed
// in (kh, kw) order. The mask !(q < -1 || q > 1), q = x / scale_a rounded to
// x's dtype, is !(x < -bound || x > bound) with the bound of mask_bound (NaN
// keeps its gradient either way).
constexpr int kCh = 8;                                        // channels per col2im thread
template <typename T, int S>
__global__ void __launch_bounds__(kThreads) col2im_mask_kernel(const float *__restrict__ dt, const T *__restrict__ x,
                                                               ConvBwdGeom q, float bound, float norm,
                                                               __nv_bfloat16 *__restrict__ gx, float *__restrict__ sum) {
    pdl_launch_dependents();
    pdl_wait();
    const uint32_t pix = blockIdx.x * kThreads + threadIdx.x;
    const uint32_t W = static_cast<uint32_t>(q.W), hwin = static_cast<uint32_t>(q.H * q.W);
    const int64_t cgroups = (q.C + kCh - 1) / kCh;
    float tsum = 0.0f;
    if (pix < hwin) {
        const int h = static_cast<int>(pix / W), w = static_cast<int>(pix - (pix / W) * W);
        int hk[kMaxTapList], hi[kMaxTapList], wk[kMaxTapList], wj[kMaxTapList];
        const int nh = tap_list<S>(h, q.p, q.k, q.d, q.s, static_cast<int>(q.Ho), hk, hi);
        const int nw = tap_list<S>(w, q.p, q.k, q.d, q.s, static_cast<int>(q.Wo), wk, wj);
        const int64_t tstride = static_cast<int64_t>(q.k) * q.k * q.P;        // one channel further: k*k rows
        for (int64_t unit = blockIdx.y; unit < q.B * cgroups; unit += gridDim.y) {
            const int64_t b = unit / cgroups, c0 = (unit - b * cgroups) * kCh;
            const int nc = q.C - c0 < kCh ? static_cast<int>(q.C - c0) : kCh;
            const float *db = dt + b * q.Ho * q.Wo + c0 * tstride;
            // kCh channels of this pixel: each tap's kCh loads are independent
            float acc[kCh];
#pragma unroll
            for (int ci = 0; ci < kCh; ++ci) acc[ci] = 0.0f;
            for (int a = 0; a < nh; ++a) {
                for (int e = 0; e < nw; ++e) {
                    const float *dr = db + (static_cast<int64_t>(hk[a]) * q.k + wk[e]) * q.P +
                                      static_cast<int64_t>(hi[a]) * q.Wo + wj[e];
                    float v[kCh];
#pragma unroll
                    for (int ci = 0; ci < kCh; ++ci) v[ci] = ci < nc ? __ldg(dr + ci * tstride) : 0.0f;
#pragma unroll
                    for (int ci = 0; ci < kCh; ++ci) acc[ci] = __fadd_rn(acc[ci], v[ci]);
                }
            }
            const int64_t base = (b * q.C + c0) * hwin + pix;
            float xv[kCh];
#pragma unroll
            for (int ci = 0; ci < kCh; ++ci) xv[ci] = ci < nc ? ld_f32<T>(x, base + ci * static_cast<int64_t>(hwin)) : 0.0f;
#pragma unroll
            for (int ci = 0; ci < kCh; ++ci) {
                if (ci >= nc) break;
                const float y = __bfloat162float(__float2bfloat16_rn(acc[ci]));
                const float ym = __fmul_rn(y, (xv[ci] < -bound || xv[ci] > bound) ? 0.0f : 1.0f);
                const float sg = (xv[ci] > 0.0f ? 1.0f : 0.0f) - (xv[ci] < 0.0f ? 1.0f : 0.0f);
                tsum = __fadd_rn(tsum, __fmul_rn(__fmul_rn(ym, sg), norm));
                gx[base + ci * static_cast<int64_t>(hwin)] = __float2bfloat16_rn(ym);   // ym is bf16-exact
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tsum += __shfl_xor_sync(0xFFFFFFFFu, tsum, o);
    if ((threadIdx.x & 31) == 0) atomicAdd(sum, tsum);
}

template <typename T>
cudaError_t launch_col2im(const float *dt, const T *x, const ConvBwdGeom &q, float bound, float norm,
                          __nv_bfloat16 *gx, float *sum, cudaStream_t s);

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

// Grid (columns / 256, rows) for the row-mapped kernels above (rows capped
// at 65535; the kernels loop over the rest), and a flat grid of up to 16
// blocks per SM.
template <typename K, typename... Args>
cudaError_t launch_rows(K kern, int64_t cols, int64_t rows, cudaStream_t s, Args... args) {
    return launch_pdl(kern, dim3(static_cast<unsigned>((cols + kThreads - 1) / kThreads),
                                 static_cast<unsigned>(rows < 65535 ? (rows > 0 ? rows : 1) : 65535)),
                      dim3(kThreads), s, args...);
}

template <typename K, typename... Args>
cudaError_t launch_flat(K kern, int64_t work, cudaStream_t s, Args... args) {
    int64_t blocks = (work + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(kern, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), s, args...);
}

template <typename T>
cudaError_t launch_col2im(const float *dt, const T *x, const ConvBwdGeom &q, float bound, float norm,
                          __nv_bfloat16 *gx, float *sum, cudaStream_t s) {
    const int64_t cols = q.H * q.W, rows = q.B * ((q.C + kCh - 1) / kCh);
    if (q.s == 1) return launch_rows(col2im_mask_kernel<T, 1>, cols, rows, s, dt, x, q, bound, norm, gx, sum);
    if (q.s == 2) return launch_rows(col2im_mask_kernel<T, 2>, cols, rows, s, dt, x, q, bound, norm, gx, sum);
    return launch_rows(col2im_mask_kernel<T, 0>, cols, rows, s, dt, x, q, bound, norm, gx, sum);
}

// The straight-through mask keeps x where q = x / scale_a (fp32, then rounded
// to x's dtype when that is bf16) lies in [-1, 1]. q is non-decreasing in x
// and odd, so the kept x are [-bound, bound] (and NaN), bound = the largest
// finite value v of x's dtype with q(v) <= 1: found here by bisection over
// the bit patterns of the non-negative finite values, with the same IEEE
// fp32 division and round-to-nearest-even as the definition.
float mask_bound(float scale_a, bool bf16) {
    auto value = [&](uint32_t u) {
        const uint32_t bits = bf16 ? (u << 16) : u;
        float f;
        __builtin_memcpy(&f, &bits, 4);
        return f;
    };
    auto kept = [&](uint32_t u) {
        float qv = value(u) / scale_a;
        if (bf16) qv = bf16_round_host(qv);
        return qv <= 1.0f;
    };
    uint32_t lo = 0, hi = bf16 ? 0x7F7Fu : 0x7F7FFFFFu;   // kept(0); the largest finite pattern
    if (kept(hi)) return value(hi);
    while (hi - lo > 1) {
        const uint32_t mid = lo + (hi - lo) / 2;
        if (kept(mid)) lo = mid;
        else hi = mid;
    }
    return value(lo);
}

// Pieces of the workspace. The input gradient's (g per pixel, D) and the
// weight gradient's (g rows, sign(x) im2col, partial sums) run one after the
// other on the stream, so they share the space.
struct ConvBwdPlan {
    ConvBwdGeom q;
    bool implicit;        // input gradient as one implicit GEMM (conv_dgrad.cu): no D
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
    // K splits for the weight gradient: at most one unit of work per CTA pair (76
    // pairs), so that no pair takes a second round
    const int64_t tiles = ((O + 255) / 256) * ((q.T + 223) / 224);
    int64_t sp = 76 / tiles;
    if (sp > 64) sp = 64;
    if (sp < 1) sp = 1;
    while (sp > 1 && q.P / sp < 512) --sp;                   // keep >= 8 slices per split
    pl.splits = static_cast<int>(sp);
    pl.ldp = (q.P + 64 * sp - 1) / (64 * sp) * (64 * sp);
    pl.implicit = dgrad_implicit_applies(B, C, H, W, O, k, s, p, d);
    pl.gp_off = 0;
    pl.dt_off = round_up256(static_cast<size_t>(q.P * O * 2));
    // the implicit route keeps x's codes where the gather route keeps D
    pl.dgrad_bytes = pl.dt_off + (pl.implicit ? round_up256(dgrad_codes_bytes(B, C, H, W))
                                              : round_up256(static_cast<size_t>(q.T * q.P * 4)));
    pl.go_off = 0;
    pl.u_off = round_up256(static_cast<size_t>(O * pl.ldp * 2));
    pl.part_off = pl.u_off + round_up256(static_cast<size_t>(q.T * pl.ldp * 2));
    pl.wgrad_bytes = pl.part_off + round_up256(static_cast<size_t>(sp * O * q.T * 4));
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

int bt_conv2d_backward_implicit(int64_t B, int64_t C, int64_t H, int64_t W, int64_t O, int kernel_size, int stride,
                                int padding, int dilation) {
    ConvBwdPlan pl;
    if (B < 1 || C < 1 || H < 1 || W < 1 || O < 1 || kernel_size < 1 || stride < 1 || padding < 0 || dilation < 1 ||
        !make_plan(B, C, H, W, O, kernel_size, stride, padding, dilation, pl))
        return 0;
    return pl.implicit ? 1 : 0;
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
    if (O % 8 != 0 || B > 65535 || kernel_size > 8) return BT_ERR_UNSUPPORTED;
    if (q.P > (int64_t(1) << 31) - 512 || q.T > (int64_t(1) << 24) || H * W > (int64_t(1) << 31) - 512 ||
        pl.ldp > (int64_t(1) << 31) - 512)
        return BT_ERR_UNSUPPORTED;
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
        const float norm = static_cast<float>(1.0 / std::sqrt(static_cast<double>(B) * C * H * W));
        const float bound = mask_bound(scale_a, x_dtype == BT_BF16);
        if (pl.implicit) {
            // one kernel: the taps reduced inside the tile, mask and grad_scale_a in its epilogue
            if (launch_dgrad_implicit(gp, static_cast<const uint16_t *>(wst), ldw, B, C, H, W, O, kernel_size, stride,
                                      padding, dilation, x, x_dtype, bf16_round_host(scale_w), bound, norm, grad_x,
                                      sum, dt, err, s) != cudaSuccess)
                return BT_ERR_CUDA;
        } else if (launch_tc_bf16(static_cast<const uint16_t *>(wst), ldw, gp, O, q.T, q.P, O, bf16_round_host(scale_w), dt,
                                  BT_F32, nullptr, err, s) != cudaSuccess) {
            return BT_ERR_CUDA;
        }
        const cudaError_t e = pl.implicit ? cudaSuccess :
            x_dtype == BT_F32
                ? launch_col2im(dt, static_cast<const float *>(x), q, bound, norm, static_cast<__nv_bfloat16 *>(grad_x),
                                sum, s)
                : launch_col2im(dt, static_cast<const __nv_bfloat16 *>(x), q, bound, norm,
                                static_cast<__nv_bfloat16 *>(grad_x), sum, s);
        if (e != cudaSuccess) return BT_ERR_CUDA;
    }
    if (grad_w != nullptr) {
        uint16_t *go = reinterpret_cast<uint16_t *>(ws + pl.go_off);
        uint16_t *u = reinterpret_cast<uint16_t *>(ws + pl.u_off);
        float *part = reinterpret_cast<float *>(ws + pl.part_off);
        const bool vec4 = (q.Ho * q.Wo) % 4 == 0 && aligned(g, 8);
        cudaError_t e = vec4 ? launch_rows(g_rows4_kernel, pl.ldp / 4, (q.O + kGRows - 1) / kGRows, s, g16, q, pl.ldp, go)
                             : launch_rows(g_rows_kernel, pl.ldp, (q.O + kGRows - 1) / kGRows, s, g16, q, pl.ldp, go);
        if (e == cudaSuccess)
            e = x_dtype == BT_F32
                    ? launch_rows(sign_im2col_t_kernel<float>, pl.ldp, (q.T + kTapRows - 1) / kTapRows, s,
                                  static_cast<const float *>(x), q, pl.ldp, u)
                    : launch_rows(sign_im2col_t_kernel<__nv_bfloat16>, pl.ldp, (q.T + kTapRows - 1) / kTapRows, s,
                                  static_cast<const __nv_bfloat16 *>(x), q, pl.ldp, u);
        if (e == cudaSuccess) e = launch_tc_bf16_splitk(go, pl.ldp, u, pl.ldp, O, q.T, pl.ldp, pl.splits, 1.0f, part, err, s);
        if (e == cudaSuccess)
            e = grad_w_dtype == BT_F32
                    ? launch_flat(split_sum_kernel<float>, O * q.T, s, static_cast<const float *>(part), pl.splits, O * q.T,
                                  bf16_round_host(scale_a), static_cast<float *>(grad_w))
                    : launch_flat(split_sum_kernel<__nv_bfloat16>, O * q.T, s, static_cast<const float *>(part), pl.splits,
                                  O * q.T, bf16_round_host(scale_a), static_cast<__nv_bfloat16 *>(grad_w));
        if (e != cudaSuccess) return BT_ERR_CUDA;
    }
    return BT_OK;
}

}  // extern "C"
