// W8A8 im2col + gemm convolution (banghao.live/blog/9 sections 3 and 4,
// MyQuantConv2d.forward): the input unfolded into im2col rows [P, T] (P =
// B*Ho*Wo output pixels, T = C*k*k taps, zero padding), the weight flattened
// to [O, T]; optionally SmoothQuant moves a per-column scale
// sqrt(max|rows[:, t]| / max|w[:, t]|) from the rows into the weight; both
// sides are quantized to int8 (per tensor, symmetric on [-127, 127], scale =
// max|v| / 127, torch's fake-quant rounding q = rint(v * (1 / scale))); the
// product of the dequantized values is dot(q_x, q_w) * s_x * s_w.
//
// The int8 products run on the tensor cores as bf16 x bf16 (every int8 value
// is a bf16 value, every product exact in fp32) in K splits of at most 1024
// taps, so that each split's fp32 sum (|sum| <= 1024 * 127^2 < 2^24) is exact;
// the splits are added as 32-bit integers (T <= 131072 taps keeps the total
// below 2^31) and scaled once: y = fp32(double(dot) * double(fp32(s_x * s_w))).
//
// Steps: column maxima of |rows| straight from x (each input element raises
// the maxima of the taps that read it) and of |w|; the smoothing scales and
// the quantization constants; the quantized weight [O, T'] and im2col rows
// [P, T'] (bf16, T' = T padded with zeros to the split size); the split
// products (tc_gemm.cu), each split's part stored NCHW; their sum.
#include <cmath>

#include <cuda_bf16.h>

#include "bt_device.cuh"
#include "bt_internal.h"

namespace bt {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxSplitTaps = 1024;      // taps per K split: 1024 * 127^2 < 2^24

struct Geo {
    int64_t B, C, H, W, O, Ho, Wo, P, T, Tp;   // Tp: padded taps (row length of the quantized operands)
    int k, s, p, d;
};

// Quantization constants, computed on the device.
struct QParams {
    float amax_x, amax_w;     // per-tensor maxima of the (smoothed) rows and weight
    float sx, inv_x;          // s = fp32(amax / 127), inv = fp32(1 / s) (0 when amax = 0)
    float sw, inv_w;
    float alpha;              // fp32(s_x * s_w)
};

// max that keeps a NaN (as torch.max does)
__device__ __forceinline__ float nan_max(float m, float v) { return (isnan(v) || v > m) ? v : m; }

template <typename T> __device__ __forceinline__ float to_f(const T *p, int64_t i);
template <> __device__ __forceinline__ float to_f<float>(const float *p, int64_t i) { return __ldg(p + i); }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(const __nv_bfloat16 *p, int64_t i) {
    return __bfloat162float(p[i]);
}

// act[t] = max over the im2col rows of |rows[:, t]| (as float bits; all >= 0):
// each input element raises the taps that read it. A block takes a run of
// pixel positions of one channel (blockIdx.y) over every image; each thread
// keeps the maxima of its position's taps in registers, then the block
// reduces them per tap and issues one global atomic per tap.
template <typename T, int S>
__global__ void __launch_bounds__(kThreads) colmax_x_kernel(const T *__restrict__ x, Geo g, unsigned int *__restrict__ act) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ unsigned int tmax[kMaxTapList * kMaxTapList];
    const int kk = g.k * g.k;
    const uint32_t W = static_cast<uint32_t>(g.W), hw = static_cast<uint32_t>(g.H * g.W);
    const uint32_t pix = blockIdx.x * kThreads + threadIdx.x;
    int hk[kMaxTapList], hi[kMaxTapList], wk[kMaxTapList], wj[kMaxTapList];
    int nh = 0, nw = 0;
    if (pix < hw) {
        const int h = static_cast<int>(pix / W), w = static_cast<int>(pix - (pix / W) * W);
        nh = tap_list<S>(h, g.p, g.k, g.d, g.s, static_cast<int>(g.Ho), hk, hi);
        nw = tap_list<S>(w, g.p, g.k, g.d, g.s, static_cast<int>(g.Wo), wk, wj);
    }
    for (int i = threadIdx.x; i < kk; i += kThreads) tmax[i] = 0u;
    __syncthreads();
    for (int64_t c = blockIdx.y; c < g.C; c += gridDim.y) {
        // the position's maximum over the images; every tap that reads the
        // position sees the same values
        unsigned int m = 0u;
        if (nh > 0 && nw > 0)
            for (int64_t b = 0; b < g.B; ++b) m = max(m, __float_as_uint(fabsf(to_f<T>(x, (b * g.C + c) * hw + pix))));
        if (m != 0u)
            for (int a = 0; a < nh; ++a)
                for (int e = 0; e < nw; ++e) atomicMax(&tmax[hk[a] * g.k + wk[e]], m);
        __syncthreads();
        for (int i = threadIdx.x; i < kk; i += kThreads) {
            if (tmax[i] != 0u) atomicMax(act + c * kk + i, tmax[i]);
            tmax[i] = 0u;
        }
        __syncthreads();
    }
}

// wmax[t] = max_o |w[o, t]|
template <typename T>
__global__ void __launch_bounds__(kThreads) colmax_w_kernel(const T *__restrict__ w, Geo g, unsigned int *__restrict__ wmax) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t n = g.O * g.T;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * kThreads)
        atomicMax(wmax + (i % g.T), __float_as_uint(fabsf(to_f<T>(w, i))));
}

// scale[t] = sqrt(act[t] / wmax[t]) with SmoothQuant, else 1; amax_x = max_t
// fp32(act[t] / scale[t]) (one block).
__global__ void __launch_bounds__(kThreads) scales_kernel(const unsigned int *__restrict__ act,
                                                          const unsigned int *__restrict__ wmax, Geo g, int smooth,
                                                          float *__restrict__ scale, QParams *__restrict__ qp) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ float red[kThreads];
    float m = 0.0f;
    for (int64_t t = threadIdx.x; t < g.T; t += kThreads) {
        const float a = __uint_as_float(act[t]);
        float sc = 1.0f, v = a;
        if (smooth) {
            sc = __fsqrt_rn(__fdiv_rn(a, __uint_as_float(wmax[t])));
            v = __fdiv_rn(a, sc);
        }
        scale[t] = sc;
        m = nan_max(m, v);
    }
    red[threadIdx.x] = m;
    __syncthreads();
    for (int o = kThreads / 2; o > 0; o >>= 1) {
        if (threadIdx.x < o) red[threadIdx.x] = nan_max(red[threadIdx.x], red[threadIdx.x + o]);
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const float amax = red[0];
        qp->amax_x = amax;
        qp->sx = amax != 0.0f ? __fdiv_rn(amax, 127.0f) : 0.0f;
        qp->inv_x = amax != 0.0f ? __fdiv_rn(1.0f, qp->sx) : 0.0f;
    }
}

// amax_w = max |fp32(w[o, t] * scale[t])| (float bits)
template <typename T>
__global__ void __launch_bounds__(kThreads) amax_w_kernel(const T *__restrict__ w, Geo g, const float *__restrict__ scale,
                                                          unsigned int *__restrict__ amax_w) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t n = g.O * g.T;
    float m = 0.0f;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * kThreads)
        m = nan_max(m, fabsf(__fmul_rn(to_f<T>(w, i), scale[i % g.T])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = nan_max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) atomicMax(amax_w, __float_as_uint(m));
}

__device__ __forceinline__ uint16_t quant_bf16(float v, float inv) {
    const float q = fminf(fmaxf(rintf(__fmul_rn(v, inv)), -127.0f), 127.0f);
    return static_cast<uint16_t>(__float_as_uint(q) >> 16);          // an integer |q| <= 127 is exact in bf16
}

// the weight quantized: qw[o, t] (pitch Tp, zeros past T); also finishes the
// weight's constants and alpha (thread 0 of block 0 only reads them).
template <typename T>
__global__ void __launch_bounds__(kThreads) quant_w_kernel(const T *__restrict__ w, Geo g, const float *__restrict__ scale,
                                                           const unsigned int *__restrict__ amax_w_bits,
                                                           QParams *__restrict__ qp, uint16_t *__restrict__ qw) {
    pdl_launch_dependents();
    pdl_wait();
    const float amax_w = __uint_as_float(*amax_w_bits);
    const float sw = amax_w != 0.0f ? __fdiv_rn(amax_w, 127.0f) : 0.0f;
    const float inv = amax_w != 0.0f ? __fdiv_rn(1.0f, sw) : 0.0f;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        qp->amax_w = amax_w;
        qp->sw = sw;
        qp->inv_w = inv;
        qp->alpha = __double2float_rn(__dmul_rn(static_cast<double>(qp->sx), static_cast<double>(sw)));
    }
    const int64_t n = g.O * g.Tp;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * kThreads) {
        const int64_t o = i / g.Tp, t = i - o * g.Tp;
        qw[i] = t < g.T ? quant_bf16(__fmul_rn(to_f<T>(w, o * g.T + t), scale[t]), inv) : uint16_t(0);
    }
}

// the im2col rows quantized: qx[p, t] (pitch Tp). A block takes 64 output
// pixels and the taps of 4 channels: x is gathered tap by tap with the pixels
// along the threads (reads along image rows), quantized into shared memory,
// and written pixel by pixel as runs of 4*k*k taps (a warp per pixel). The
// block's taps are tabulated once (channel, offsets, scale), so the loops
// divide nothing; without SmoothQuant the scale is 1 and v / 1 = v is not
// computed. The block of the last channel group also zeroes the padding taps
// [T, Tp).
constexpr int kQP = 64, kQC = 4, kQT = kQC * kMaxTapList * kMaxTapList;
template <typename T, bool SMOOTH>
__global__ void __launch_bounds__(kThreads) quant_rows_kernel(const T *__restrict__ x, Geo g, const float *__restrict__ scale,
                                                              const QParams *__restrict__ qp, uint16_t *__restrict__ qx) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ uint16_t tile[kQP][kQT + 2];
    __shared__ int pb[kQP], ph[kQP], pw[kQP];
    __shared__ int toff[kQT], th[kQT], tw[kQT];
    __shared__ float ts[kQT];
    const float inv = qp->inv_x;
    const int64_t p0 = static_cast<int64_t>(blockIdx.x) * kQP;
    const int c0 = static_cast<int>(blockIdx.y) * kQC;
    const int kk = g.k * g.k;
    const int nc = g.C - c0 < kQC ? static_cast<int>(g.C - c0) : kQC;
    const int ntaps = nc * kk;
    if (threadIdx.x < kQP) {
        const int64_t p = p0 + threadIdx.x;
        int b = -1, h0 = 0, w0 = 0;
        if (p < g.P) {
            const uint32_t hwo = static_cast<uint32_t>(g.Ho * g.Wo), wo = static_cast<uint32_t>(g.Wo);
            const uint32_t bb = static_cast<uint32_t>(p / hwo), pix = static_cast<uint32_t>(p - static_cast<int64_t>(bb) * hwo);
            const uint32_t oi = pix / wo, oj = pix - oi * wo;
            b = static_cast<int>(bb);
            h0 = static_cast<int>(oi) * g.s - g.p;
            w0 = static_cast<int>(oj) * g.s - g.p;
        }
        pb[threadIdx.x] = b;
        ph[threadIdx.x] = h0;
        pw[threadIdx.x] = w0;
    }
    for (int tt = threadIdx.x; tt < ntaps; tt += kThreads) {
        const int ci = tt / kk, tap = tt - ci * kk, kh = tap / g.k, kw = tap - kh * g.k;
        toff[tt] = (c0 + ci) * static_cast<int>(g.H * g.W) + kh * g.d * static_cast<int>(g.W) + kw * g.d;
        th[tt] = kh * g.d;
        tw[tt] = kw * g.d;
        ts[tt] = SMOOTH ? scale[(c0 + ci) * kk + tap] : 1.0f;
    }
    __syncthreads();
    const int pp = threadIdx.x & (kQP - 1);
    const int b = pb[pp], h0 = ph[pp], w0 = pw[pp];
    // the pixel's image and window corner; per tap only the offset within the image
    const T *xi = x + (b >= 0 ? static_cast<int64_t>(b) * g.C * g.H * g.W : 0);
    const int corner = h0 * static_cast<int>(g.W) + w0;
    const int H = static_cast<int>(g.H), W = static_cast<int>(g.W);
    for (int tt = threadIdx.x / kQP; tt < ntaps; tt += kThreads / kQP) {
        uint16_t v = 0;
        if (b >= 0) {
            const int ih = h0 + th[tt], iw = w0 + tw[tt];
            float xv = 0.0f;
            if (static_cast<unsigned>(ih) < static_cast<unsigned>(H) && static_cast<unsigned>(iw) < static_cast<unsigned>(W))
                xv = to_f<T>(xi, corner + toff[tt]);
            v = quant_bf16(SMOOTH ? __fdiv_rn(xv, ts[tt]) : xv, inv);
        }
        tile[pp][tt] = v;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int q = warp; q < kQP; q += kThreads / 32) {
        const int64_t p = p0 + q;
        if (p >= g.P) break;
        uint16_t *row = qx + p * g.Tp + static_cast<int64_t>(c0) * kk;
        for (int tt = lane; tt < ntaps; tt += 32) row[tt] = tile[q][tt];
        if (c0 + kQC >= g.C)
            for (int64_t t = g.T + lane; t < g.Tp; t += 32) qx[p * g.Tp + t] = 0;
    }
}

// out[i] = fp32(double(sum over splits of part[s][i]) * alpha), the parts laid
// out NCHW like the output: the partial sums are integers below 2^24, added
// exactly as 32-bit integers; while |sum| <= 2^24 the sum is exact in fp32 and
// sum * alpha (48 bits) exact in double, so one fp32 multiply gives the same
// result, and only larger sums take the double product.
__device__ __forceinline__ float scale_dot(int acc, float alphaf) {
    if (acc <= (1 << 24) && acc >= -(1 << 24)) return __fmul_rn(static_cast<float>(acc), alphaf);
    return __double2float_rn(__dmul_rn(static_cast<double>(acc), static_cast<double>(alphaf)));
}

template <typename O>
__global__ void __launch_bounds__(kThreads) combine_kernel(const float *__restrict__ part, int splits, int64_t n,
                                                           const QParams *__restrict__ qp, O *__restrict__ out) {
    pdl_launch_dependents();
    pdl_wait();
    const float alphaf = qp->alpha;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * kThreads) {
        int acc = 0;
        for (int s = 0; s < splits; ++s) acc += __float2int_rn(__ldg(part + s * n + i));
        const float y = scale_dot(acc, alphaf);
        if constexpr (sizeof(O) == 4) out[i] = y;
        else out[i] = __float2bfloat16_rn(y);
    }
}

template <typename K, typename... Args>
cudaError_t launch(K kern, dim3 grid, cudaStream_t s, Args... args) {
    return launch_pdl(kern, grid, dim3(kThreads), s, args...);
}

unsigned flat_blocks(int64_t n) {
    int64_t b = (n + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    return static_cast<unsigned>(b < 1 ? 1 : (b > cap ? cap : b));
}
unsigned rows_cap(int64_t rows) { return static_cast<unsigned>(rows < 1 ? 1 : (rows > 65535 ? 65535 : rows)); }

bool make_geo(int64_t B, int64_t C, int64_t H, int64_t W, int64_t O, int k, int s, int p, int d, Geo &g, int &splits) {
    g.B = B; g.C = C; g.H = H; g.W = W; g.O = O; g.k = k; g.s = s; g.p = p; g.d = d;
    const int64_t hn = H + 2 * static_cast<int64_t>(p) - static_cast<int64_t>(d) * (k - 1) - 1;
    const int64_t wn = W + 2 * static_cast<int64_t>(p) - static_cast<int64_t>(d) * (k - 1) - 1;
    if (hn < 0 || wn < 0) return false;
    g.Ho = hn / s + 1;
    g.Wo = wn / s + 1;
    g.P = B * g.Ho * g.Wo;
    g.T = C * k * k;
    splits = static_cast<int>((g.T + kMaxSplitTaps - 1) / kMaxSplitTaps);
    if (splits < 1) splits = 1;
    const int64_t unit = 64 * static_cast<int64_t>(splits);
    g.Tp = (g.T + unit - 1) / unit * unit;
    return true;
}

struct Layout {
    size_t act, wmax, amax_w, qp, scale, qw, qx, part, total;
};

Layout layout(const Geo &g, int splits) {
    Layout l{};
    size_t o = 0;
    l.act = o; o += round_up256(static_cast<size_t>(g.T) * 4);
    l.wmax = o; o += round_up256(static_cast<size_t>(g.T) * 4);
    l.amax_w = o; o += 256;
    l.qp = o; o += 256;
    l.scale = o; o += round_up256(static_cast<size_t>(g.T) * 4);
    l.qw = o; o += round_up256(static_cast<size_t>(g.O * g.Tp) * 2);
    l.qx = o; o += round_up256(static_cast<size_t>(g.P * g.Tp) * 2);
    l.part = o; o += round_up256(static_cast<size_t>(splits) * g.O * g.P * 4);
    l.total = o;
    return l;
}

template <typename TX, typename TW>
cudaError_t run(const TX *x, const TW *w, const Geo &g, int splits, int smooth, void *out, bt_dtype out_t, uint8_t *ws,
                unsigned int *err, cudaStream_t s) {
    const Layout l = layout(g, splits);
    unsigned int *act = reinterpret_cast<unsigned int *>(ws + l.act);
    unsigned int *wmax = reinterpret_cast<unsigned int *>(ws + l.wmax);
    unsigned int *amax_w = reinterpret_cast<unsigned int *>(ws + l.amax_w);
    QParams *qp = reinterpret_cast<QParams *>(ws + l.qp);
    float *scale = reinterpret_cast<float *>(ws + l.scale);
    uint16_t *qw = reinterpret_cast<uint16_t *>(ws + l.qw);
    uint16_t *qx = reinterpret_cast<uint16_t *>(ws + l.qx);
    float *part = reinterpret_cast<float *>(ws + l.part);
    cudaError_t e = cudaMemsetAsync(ws, 0, l.scale, s);            // act, wmax, amax_w, qp
    const dim3 pix_grid(static_cast<unsigned>((g.H * g.W + kThreads - 1) / kThreads), rows_cap(g.C));
    if (e == cudaSuccess) {
        if (g.s == 1) e = launch(colmax_x_kernel<TX, 1>, pix_grid, s, x, g, act);
        else if (g.s == 2) e = launch(colmax_x_kernel<TX, 2>, pix_grid, s, x, g, act);
        else e = launch(colmax_x_kernel<TX, 0>, pix_grid, s, x, g, act);
    }
    if (e == cudaSuccess) e = launch(colmax_w_kernel<TW>, dim3(flat_blocks(g.O * g.T)), s, w, g, wmax);
    if (e == cudaSuccess)
        e = launch(scales_kernel, dim3(1), s, static_cast<const unsigned int *>(act), static_cast<const unsigned int *>(wmax),
                   g, smooth, scale, qp);
    if (e == cudaSuccess)
        e = launch(amax_w_kernel<TW>, dim3(flat_blocks(g.O * g.T)), s, w, g, static_cast<const float *>(scale), amax_w);
    if (e == cudaSuccess)
        e = launch(quant_w_kernel<TW>, dim3(flat_blocks(g.O * g.Tp)), s, w, g, static_cast<const float *>(scale),
                   static_cast<const unsigned int *>(amax_w), qp, qw);
    if (e == cudaSuccess) {
        const dim3 qgrid(static_cast<unsigned>((g.P + kQP - 1) / kQP), static_cast<unsigned>((g.C + kQC - 1) / kQC));
        e = smooth ? launch(quant_rows_kernel<TX, true>, qgrid, s, x, g, static_cast<const float *>(scale),
                            static_cast<const QParams *>(qp), qx)
                   : launch(quant_rows_kernel<TX, false>, qgrid, s, x, g, static_cast<const float *>(scale),
                            static_cast<const QParams *>(qp), qx);
    }
    if (e == cudaSuccess)
        e = launch_tc_bf16_splitk(qw, g.Tp, qx, g.Tp, g.O, g.P, g.Tp, splits, 1.0f, part, err, s, g.Ho * g.Wo);
    if (e == cudaSuccess) {
        const int64_t n = g.B * g.O * g.Ho * g.Wo;
        const dim3 grid(flat_blocks(n));
        e = out_t == BT_F32 ? launch(combine_kernel<float>, grid, s, static_cast<const float *>(part), splits, n,
                                     static_cast<const QParams *>(qp), static_cast<float *>(out))
                            : launch(combine_kernel<__nv_bfloat16>, grid, s, static_cast<const float *>(part), splits, n,
                                     static_cast<const QParams *>(qp), static_cast<__nv_bfloat16 *>(out));
    }
    return e;
}

}  // namespace
}  // namespace bt

using namespace bt;

extern "C" {

size_t bt_w8a8_conv2d_workspace(int64_t B, int64_t C, int64_t H, int64_t W, int64_t O, int kernel_size, int stride,
                                int padding, int dilation) {
    Geo g;
    int splits = 1;
    if (B < 0 || C < 1 || H < 1 || W < 1 || O < 1 || kernel_size < 1 || stride < 1 || padding < 0 || dilation < 1 ||
        !make_geo(B, C, H, W, O, kernel_size, stride, padding, dilation, g, splits))
        return 0;
    return layout(g, splits).total;
}

bt_status bt_w8a8_conv2d(const void *x, bt_dtype x_dtype, const void *w, bt_dtype w_dtype, int64_t B, int64_t C,
                         int64_t H, int64_t W, int64_t O, int kernel_size, int stride, int padding, int dilation,
                         int smooth, void *out, bt_dtype out_dtype, void *workspace, size_t workspace_bytes,
                         bt_stream stream) {
    if ((x_dtype != BT_F32 && x_dtype != BT_BF16) || (w_dtype != BT_F32 && w_dtype != BT_BF16)) return BT_ERR_INVALID_ARG;
    if (out_dtype != BT_F32 && out_dtype != BT_BF16) return BT_ERR_INVALID_ARG;
    if (B < 0 || C < 1 || H < 1 || W < 1 || O < 1 || kernel_size < 1 || stride < 1 || padding < 0 || dilation < 1)
        return BT_ERR_INVALID_ARG;
    Geo g;
    int splits = 1;
    if (!make_geo(B, C, H, W, O, kernel_size, stride, padding, dilation, g, splits)) return BT_ERR_INVALID_ARG;
    if (kernel_size > kMaxTapList || H * W > (int64_t(1) << 31) - 512 || g.Ho * g.Wo > (int64_t(1) << 31) - 512 ||
        g.P > (int64_t(1) << 31) - 512 || g.T > 131072 || O > (int64_t(1) << 24) ||
        C * H * W > (int64_t(1) << 31) - 1)
        return BT_ERR_UNSUPPORTED;
    if (B == 0) return BT_OK;
    if (x == nullptr || w == nullptr || out == nullptr) return BT_ERR_INVALID_ARG;
    if (!tc_available()) return BT_ERR_UNSUPPORTED;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(out, 16)) return BT_ERR_ALIGNMENT;
    const size_t need = layout(g, splits).total;
    if (workspace == nullptr || workspace_bytes < need) return BT_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return BT_ERR_ALIGNMENT;
    unsigned int *err = device_error_word();
    if (err == nullptr) return BT_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    cudaError_t e;
    if (x_dtype == BT_F32)
        e = w_dtype == BT_F32 ? run(static_cast<const float *>(x), static_cast<const float *>(w), g, splits, smooth, out,
                                    out_dtype, ws, err, s)
                              : run(static_cast<const float *>(x), static_cast<const __nv_bfloat16 *>(w), g, splits,
                                    smooth, out, out_dtype, ws, err, s);
    else
        e = w_dtype == BT_F32 ? run(static_cast<const __nv_bfloat16 *>(x), static_cast<const float *>(w), g, splits,
                                    smooth, out, out_dtype, ws, err, s)
                              : run(static_cast<const __nv_bfloat16 *>(x), static_cast<const __nv_bfloat16 *>(w), g,
                                    splits, smooth, out, out_dtype, ws, err, s);
    return e == cudaSuccess ? BT_OK : BT_ERR_CUDA;
}

}  // extern "C"
