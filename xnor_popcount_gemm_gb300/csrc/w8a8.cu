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
#include <cstdlib>
#include <cstring>
#include <type_traits>

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

__device__ __forceinline__ float as_f(float v) { return v; }
__device__ __forceinline__ float as_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T zero_of();
template <> __device__ __forceinline__ float zero_of<float>() { return 0.0f; }
template <> __device__ __forceinline__ __nv_bfloat16 zero_of<__nv_bfloat16>() { return __ushort_as_bfloat16(0); }

// act[t] = max over the im2col rows of |rows[:, t]| (as float bits; all >= 0):
// each input element raises the taps that read it. A block takes a run of
// pixel positions of one channel (blockIdx.y) over a group of images
// (blockIdx.z); each thread keeps the maximum of its position over the group
// (sixteen loads in flight), raises its taps in shared memory, and the block
// issues one global atomic per tap.
template <typename T, int S>
__global__ void __launch_bounds__(kThreads) colmax_x_kernel(const T *__restrict__ x, Geo g, int imgs_per_group,
                                                            unsigned int *__restrict__ act) {
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
    const int64_t b0 = static_cast<int64_t>(blockIdx.z) * imgs_per_group;
    const int64_t b1 = b0 + imgs_per_group < g.B ? b0 + imgs_per_group : g.B;
    for (int i = threadIdx.x; i < kk; i += kThreads) tmax[i] = 0u;
    __syncthreads();
    for (int64_t c = blockIdx.y; c < g.C; c += gridDim.y) {
        // the position's maximum over the group's images; every tap that
        // reads the position sees the same values
        unsigned int m = 0u;
        if (nh > 0 && nw > 0) {
            const T *src = x + (b0 * g.C + c) * hw + pix;
            const int64_t img = g.C * hw;
            int64_t b = b0;
            for (; b + 16 <= b1; b += 16, src += 16 * img) {
                float v[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) v[u] = to_f<T>(src, u * img);
#pragma unroll
                for (int u = 0; u < 16; ++u) m = max(m, __float_as_uint(fabsf(v[u])));
            }
            for (; b < b1; ++b, src += img) m = max(m, __float_as_uint(fabsf(to_f<T>(src, 0))));
        }
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

// Geometry of the staged quantize-unfold: a unit is (image, band of R output
// rows, range of Wc output columns, CC channels); its NR x NW input window per
// channel (zeros outside the image and past the last channel) is staged in
// shared memory, so the gather reads only shared memory and every global
// access is a coalesced run.
struct QTile {
    int R, Wc, nb, nwc;   // output rows per band, columns per range; bands, ranges
    int NR, NW, E;        // staged rows, columns, and NR * NW
    int CC, TB, pitch;    // channels per unit, taps per unit row (CC * k * k), tile row pitch (elements)
    int ncu;              // channel units: ceil(C / CC)
    int qbits;            // log2 of the pixel slots per unit (R * Wc <= 1 << qbits)
    int64_t T8;           // T rounded up to 8 taps
    FastDiv div_e, div_nw, div_kk, div_k, div_wc, div_ncu, div_nwc, div_nb;
    FastDiv div_chk, div_chk_last;   // 16-byte chunks of a unit row: TB / 8, and in the last channel unit
};
constexpr int kStageItems = 3;   // window items (8 channels at one position) per thread

// q = clamp(rint(fp32(v * inv)), -127, 127) for two values, as a pair of bf16
// codes. Adding and subtracting 1.5 * 2^23 rounds the product to an integer,
// ties to even, for |product| < 2^22, exactly as rint; larger products,
// infinities and NaN leave the clamp as +-127 just as they do after rint (NaN
// as -127, like fmaxf(NaN, -127)); the clamped integers are exact in bf16. A
// product in (-0.5, 0] gives +0 where rint gives -0: the same zero in every
// product it enters.
__device__ __forceinline__ uint32_t quant_pair(float v0, float v1, float inv) {
    constexpr float kRound = 12582912.0f;
    const float r0 = __fsub_rn(__fadd_rn(__fmul_rn(v0, inv), kRound), kRound);
    const float r1 = __fsub_rn(__fadd_rn(__fmul_rn(v1, inv), kRound), kRound);
    const __nv_bfloat162 q = __hmin2(__hmax2(__floats2bfloat162_rn(r0, r1), __float2bfloat162_rn(-127.0f)),
                                     __float2bfloat162_rn(127.0f));
    return *reinterpret_cast<const uint32_t *>(&q);
}

// the unit's quantized rows: qx[p, c0*k*k .. +CC*k*k) for its pixels p, and,
// for the last channel unit, zeros over [T, Tp). Stage 1 copies the window
// (its loads issued before the wait on the previous kernel: x is an input of
// the whole call); without SmoothQuant a code depends on the value alone, so
// the window holds codes, each quantized once however many taps read it;
// with SmoothQuant it holds x and the taps are quantized in stage 2. Stage 2
// gathers 8 taps of one pixel per thread, the pixels along the lanes (the
// window read at a stride of s elements, the tile written with 16-byte
// stores at an odd 16-byte pitch); stage 3 writes the runs of taps with
// 16-byte stores, consecutive threads on consecutive chunks. Shared memory:
// tile [1 << qbits][pitch] u16, tap byte offsets [TB] int, pixel corner
// (bytes) and row [1 << qbits] int each, scales [TB] f32 (SmoothQuant),
// window [CC][NR][NW] (u16 codes, or T with SmoothQuant).
template <typename T, bool SMOOTH>
__global__ void __launch_bounds__(kThreads, 5) quant_tile_kernel(const T *__restrict__ x, Geo g, QTile u,
                                                              const float *__restrict__ scale,
                                                              const QParams *__restrict__ qp, uint16_t *__restrict__ qx) {
    using WT = typename std::conditional<SMOOTH, T, uint16_t>::type;
    pdl_launch_dependents();
    extern __shared__ __align__(16) uint8_t qsm[];
    const int slots = 1 << u.qbits;
    uint16_t *tile = reinterpret_cast<uint16_t *>(qsm);
    int *coff = reinterpret_cast<int *>(tile + slots * u.pitch);
    int *corner = coff + u.TB;
    int *prow = corner + slots;
    float *ts = reinterpret_cast<float *>(prow + slots);
    WT *win = reinterpret_cast<WT *>(ts + (SMOOTH ? u.TB : 0));

    const int tid = threadIdx.x;
    const int kk = g.k * g.k;
    // the channel units of the same pixels run one after another, so that
    // each row of qx is written as a whole within a short time
    const uint32_t unit = fdiv(blockIdx.x, u.div_ncu), cu = blockIdx.x - unit * static_cast<uint32_t>(u.ncu);
    const uint32_t rb = fdiv(unit, u.div_nwc), range = unit - rb * static_cast<uint32_t>(u.nwc);
    const uint32_t b32 = fdiv(rb, u.div_nb), band = rb - b32 * static_cast<uint32_t>(u.nb);
    const int64_t b = b32;
    const int i0 = static_cast<int>(band) * u.R, j0 = static_cast<int>(range) * u.Wc;
    const int c0 = static_cast<int>(cu) * u.CC;
    const int nc = g.C - c0 < u.CC ? static_cast<int>(g.C - c0) : u.CC;
    // window origin (may be negative: padding) and 32-bit offsets within the
    // unit's first channel plane (C * H * W < 2^31)
    const int ih0 = i0 * g.s - g.p, iw0 = j0 * g.s - g.p;
    const int H = static_cast<int>(g.H), W = static_cast<int>(g.W), hw = H * W;
    const T *xc = x + (b * g.C + c0) * g.H * g.W;

    // stage 1: the window, win[ci][r][c] from x[b, c0 + ci, ih0 + r, iw0 + c].
    // Items (8-channel group, window position), positions along the threads;
    // every thread issues the loads of all its items (at most kStageItems)
    // before using any, so that each waits for one round trip.
    const int nitems = u.E * (u.CC / 8);
    T v[kStageItems][8];
    int dst[kStageItems];
#pragma unroll
    for (int j = 0; j < kStageItems; ++j) {
        const int it = tid + j * kThreads;
        dst[j] = -1;
        if (it < nitems) {
            const int cg = static_cast<int>(fdiv(static_cast<uint32_t>(it), u.div_e));
            const int e = it - cg * u.E;
            const int r = static_cast<int>(fdiv(static_cast<uint32_t>(e), u.div_nw)), c = e - r * u.NW;
            const int ih = ih0 + r, iw = iw0 + c;
            const bool inside = static_cast<unsigned>(ih) < static_cast<unsigned>(H) &&
                                static_cast<unsigned>(iw) < static_cast<unsigned>(W);
            const int off = 8 * cg * hw + (inside ? ih * W + iw : 0);
#pragma unroll
            for (int h = 0; h < 8; ++h) v[j][h] = (inside && 8 * cg + h < nc) ? xc[off + h * hw] : zero_of<T>();
            dst[j] = 8 * cg * u.E + e;
        }
    }
    // tap byte offsets within the window, pixel corners and output rows
    for (int tt = tid; tt < u.TB; tt += kThreads) {
        const int ci = static_cast<int>(fdiv(static_cast<uint32_t>(tt), u.div_kk)), tap = tt - ci * kk;
        const int kh = static_cast<int>(fdiv(static_cast<uint32_t>(tap), u.div_k)), kw = tap - kh * g.k;
        coff[tt] = (ci * u.E + kh * g.d * u.NW + kw * g.d) * static_cast<int>(sizeof(WT));
    }
    if (tid < slots) {
        const int qi = static_cast<int>(fdiv(static_cast<uint32_t>(tid), u.div_wc)), qj = tid - qi * u.Wc;
        const bool ok = tid < u.R * u.Wc && i0 + qi < g.Ho && j0 + qj < g.Wo;
        corner[tid] = ok ? (qi * g.s * u.NW + qj * g.s) * static_cast<int>(sizeof(WT)) : 0;
        prow[tid] = ok ? static_cast<int>((b * g.Ho + i0 + qi) * g.Wo + j0 + qj) : -1;
    }
    pdl_wait();
    const float inv = qp->inv_x;
#pragma unroll
    for (int j = 0; j < kStageItems; ++j)
        if (dst[j] >= 0) {
            if constexpr (SMOOTH) {
#pragma unroll
                for (int h = 0; h < 8; ++h) win[dst[j] + h * u.E] = v[j][h];
            } else {
#pragma unroll
                for (int h = 0; h < 8; h += 2) {
                    const uint32_t q2 = quant_pair(as_f(v[j][h]), as_f(v[j][h + 1]), inv);
                    win[dst[j] + h * u.E] = static_cast<uint16_t>(q2);
                    win[dst[j] + (h + 1) * u.E] = static_cast<uint16_t>(q2 >> 16);
                }
            }
        }
    if constexpr (SMOOTH)
        for (int tt = tid; tt < u.TB; tt += kThreads)
            ts[tt] = tt < nc * kk ? scale[static_cast<int64_t>(c0) * kk + tt] : 1.0f;
    const bool last = c0 + u.CC >= g.C;
    const int nchk = last ? static_cast<int>((u.T8 - static_cast<int64_t>(c0) * kk) / 8) : u.TB / 8;
    __syncthreads();

    // stage 2: the tile, 8 taps of pixel q per item
    {
        const int q = tid & (slots - 1);
        const uint8_t *wq = reinterpret_cast<const uint8_t *>(win) + corner[q];
        if (prow[q] >= 0)
            for (int ch = tid >> u.qbits; ch < nchk; ch += kThreads >> u.qbits) {
                const int4 oa = *reinterpret_cast<const int4 *>(coff + ch * 8);
                const int4 ob = *reinterpret_cast<const int4 *>(coff + ch * 8 + 4);
                const int o[8] = {oa.x, oa.y, oa.z, oa.w, ob.x, ob.y, ob.z, ob.w};
                uint32_t wv[4];
                if constexpr (SMOOTH) {
                    const float4 sa = *reinterpret_cast<const float4 *>(ts + ch * 8);
                    const float4 sb = *reinterpret_cast<const float4 *>(ts + ch * 8 + 4);
                    const float sc[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h)
                        wv[h] = quant_pair(__fdiv_rn(as_f(*reinterpret_cast<const T *>(wq + o[2 * h])), sc[2 * h]),
                                           __fdiv_rn(as_f(*reinterpret_cast<const T *>(wq + o[2 * h + 1])), sc[2 * h + 1]),
                                           inv);
                } else {
#pragma unroll
                    for (int h = 0; h < 4; ++h)
                        wv[h] = static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(wq + o[2 * h])) |
                                (static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(wq + o[2 * h + 1])) << 16);
                }
                *reinterpret_cast<uint4 *>(tile + q * u.pitch + ch * 8) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
    }
    __syncthreads();

    // stage 3: the pixels' runs of taps, items (pixel, 16-byte chunk), then
    // the zero tail past T
    const FastDiv dchk = last ? u.div_chk_last : u.div_chk;
    const int npix = u.R * u.Wc;
    for (int i = tid; i < npix * nchk; i += kThreads) {
        const int q = static_cast<int>(fdiv(static_cast<uint32_t>(i), dchk)), ch = i - q * nchk;
        const int pr = prow[q];
        if (pr >= 0)
            *reinterpret_cast<uint4 *>(qx + static_cast<int64_t>(pr) * g.Tp + c0 * kk + ch * 8) =
                *reinterpret_cast<const uint4 *>(tile + q * u.pitch + ch * 8);
    }
    if (last && u.T8 < g.Tp) {
        const int warp = tid >> 5, lane = tid & 31;
        for (int q = warp; q < npix; q += kThreads / 32) {
            const int pr = prow[q];
            if (pr < 0) continue;
            uint16_t *row = qx + static_cast<int64_t>(pr) * g.Tp;
            for (int64_t t = u.T8 + lane * 8; t < g.Tp; t += 256) *reinterpret_cast<uint4 *>(row + t) = make_uint4(0, 0, 0, 0);
        }
    }
}

// bytes of shared memory the staged unfold needs for plan u and window element size es
size_t qtile_smem(const QTile &u, int es, bool smooth) {
    const size_t slots = size_t(1) << u.qbits;
    return slots * u.pitch * 2 + static_cast<size_t>(u.TB) * 4 + slots * 8 + (smooth ? static_cast<size_t>(u.TB) * 4 : 0) +
           static_cast<size_t>(u.CC) * u.E * es;
}

// The staged unfold's plan: 16 channels (more for small kernels, up to ~144
// taps a row, at most the channel count rounded up to 16) and 64 pixel slots
// (fewer while the tile passes 28 KB); a band of whole output rows where Wo
// fits, else a range of columns; the window shrinks (rows, then columns)
// until it fits 16 KB and kStageItems items per thread. False: no plan fits
// (very large dilation), and the direct gather takes the call.
bool plan_qtile(const Geo &g, int es, QTile &u) {
    const int kk = g.k * g.k;
    // 32-bit window coordinates and offsets within an image
    if (g.H + 2 * static_cast<int64_t>(g.p) >= (int64_t(1) << 30) || g.W + 2 * static_cast<int64_t>(g.p) >= (int64_t(1) << 30))
        return false;
    u.CC = 144 / kk / 16 * 16;
    if (u.CC < 16) u.CC = 16;
    if (u.CC > (g.C + 15) / 16 * 16) u.CC = static_cast<int>((g.C + 15) / 16 * 16);
    if ((g.C + u.CC) * g.H * g.W >= (int64_t(1) << 31)) return false;
    u.TB = u.CC * kk;
    u.pitch = ((u.TB / 8) & 1) ? u.TB : u.TB + 8;
    u.qbits = 6;
    while (u.qbits > 3 && (int64_t(1) << u.qbits) * u.pitch * 2 > 28 * 1024) --u.qbits;
    if ((int64_t(1) << u.qbits) * u.pitch * 2 > 28 * 1024) return false;
    const int64_t slots = int64_t(1) << u.qbits;
    int64_t Wc = g.Wo < slots ? g.Wo : slots;
    int64_t nwc = (g.Wo + Wc - 1) / Wc;
    Wc = (g.Wo + nwc - 1) / nwc;
    int64_t nb = (g.Ho + slots / Wc - 1) / (slots / Wc);
    int64_t R = (g.Ho + nb - 1) / nb;
    const int64_t reach = static_cast<int64_t>(g.k - 1) * g.d + 1;
    for (;;) {
        const int64_t NR = (R - 1) * g.s + reach, NW = (Wc - 1) * g.s + reach;
        const int64_t E = NR * NW;
        if (E * u.CC * es <= 16 * 1024 && E * (u.CC / 8) <= kStageItems * kThreads) {
            u.R = static_cast<int>(R);
            u.Wc = static_cast<int>(Wc);
            u.nb = static_cast<int>((g.Ho + R - 1) / R);
            u.nwc = static_cast<int>((g.Wo + Wc - 1) / Wc);
            u.NR = static_cast<int>(NR);
            u.NW = static_cast<int>(NW);
            u.E = static_cast<int>(E);
            u.T8 = (g.T + 7) / 8 * 8;
            u.ncu = static_cast<int>((g.C + u.CC - 1) / u.CC);
            u.div_e = make_fastdiv(static_cast<uint32_t>(E));
            u.div_nw = make_fastdiv(static_cast<uint32_t>(NW));
            u.div_kk = make_fastdiv(static_cast<uint32_t>(kk));
            u.div_k = make_fastdiv(static_cast<uint32_t>(g.k));
            u.div_wc = make_fastdiv(static_cast<uint32_t>(Wc));
            u.div_ncu = make_fastdiv(static_cast<uint32_t>(u.ncu));
            u.div_nwc = make_fastdiv(static_cast<uint32_t>(u.nwc));
            u.div_nb = make_fastdiv(static_cast<uint32_t>(u.nb));
            u.div_chk = make_fastdiv(static_cast<uint32_t>(u.TB / 8));
            const int64_t last_chk = (u.T8 - (u.ncu - 1) * static_cast<int64_t>(u.CC) * kk) / 8;
            u.div_chk_last = make_fastdiv(static_cast<uint32_t>(last_chk > 0 ? last_chk : 1));
            return g.B * u.nb * u.nwc * u.ncu < (int64_t(1) << 31);
        }
        if (R > 1) R = (R + 1) / 2;
        else if (Wc > 1) Wc = (Wc + 1) / 2;
        else return false;
    }
}

// The direct gather, for geometries no staged plan fits: the im2col rows
// quantized, qx[p, t] (pitch Tp). A block takes 64 output
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
// (The double product is a call of its own, so that the common case runs no
// double-precision instruction at all.)
__device__ __noinline__ float scale_dot_wide(int acc, float alphaf) {
    return __double2float_rn(__dmul_rn(static_cast<double>(acc), static_cast<double>(alphaf)));
}
__device__ __forceinline__ float scale_dot(int acc, float alphaf) {
    if (acc <= (1 << 24) && acc >= -(1 << 24)) return __fmul_rn(static_cast<float>(acc), alphaf);
    return scale_dot_wide(acc, alphaf);
}

template <typename O>
__device__ __forceinline__ void store4(O *out, int64_t i4, float y0, float y1, float y2, float y3) {
    if constexpr (sizeof(O) == 4) {
        reinterpret_cast<float4 *>(out)[i4] = make_float4(y0, y1, y2, y3);
    } else {
        const __nv_bfloat162 a = __floats2bfloat162_rn(y0, y1), c = __floats2bfloat162_rn(y2, y3);
        uint2 v;
        v.x = *reinterpret_cast<const uint32_t *>(&a);
        v.y = *reinterpret_cast<const uint32_t *>(&c);
        reinterpret_cast<uint2 *>(out)[i4] = v;
    }
}

// Four elements per 16-byte load when n is a multiple of 4 (each part then
// starts 16-byte aligned), four such groups per thread with all their loads
// issued first (SPL = the number of parts when 1 to 4); else one element at
// a time.
template <typename O, int SPL>
__global__ void __launch_bounds__(kThreads) combine_kernel(const float *__restrict__ part, int splits, int64_t n,
                                                           const QParams *__restrict__ qp, O *__restrict__ out) {
    pdl_launch_dependents();
    pdl_wait();
    const float alphaf = qp->alpha;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    if (SPL > 0 && (n & 3) == 0) {
        constexpr int U = 4, S = SPL > 0 ? SPL : 1;
        const int64_t n4 = n >> 2;
        const float4 *p4 = reinterpret_cast<const float4 *>(part);
        for (int64_t i0 = first; i0 < n4; i0 += U * stride) {
            float4 v[U][S];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int sp = 0; sp < S; ++sp)
                    v[u][sp] = i0 + u * stride < n4 ? __ldg(p4 + sp * n4 + i0 + u * stride) : make_float4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (i0 + u * stride >= n4) break;
                int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
                for (int sp = 0; sp < S; ++sp) {
                    a0 += __float2int_rn(v[u][sp].x);
                    a1 += __float2int_rn(v[u][sp].y);
                    a2 += __float2int_rn(v[u][sp].z);
                    a3 += __float2int_rn(v[u][sp].w);
                }
                store4(out, i0 + u * stride, scale_dot(a0, alphaf), scale_dot(a1, alphaf), scale_dot(a2, alphaf),
                       scale_dot(a3, alphaf));
            }
        }
        return;
    }
    for (int64_t i = first; i < n; i += stride) {
        int acc = 0;
        for (int s = 0; s < splits; ++s) acc += __float2int_rn(__ldg(part + s * n + i));
        const float y = scale_dot(acc, alphaf);
        if constexpr (sizeof(O) == 4) out[i] = y;
        else out[i] = __float2bfloat16_rn(y);
    }
}

template <typename O>
cudaError_t launch_combine(const float *part, int splits, int64_t n, const QParams *qp, O *out, cudaStream_t s);

template <typename K, typename... Args>
cudaError_t launch(K kern, dim3 grid, cudaStream_t s, Args... args) {
    return launch_pdl(kern, grid, dim3(kThreads), s, args...);
}

unsigned flat_blocks(int64_t n) {
    int64_t b = (n + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    return static_cast<unsigned>(b < 1 ? 1 : (b > cap ? cap : b));
}
template <typename O>
cudaError_t launch_combine(const float *part, int splits, int64_t n, const QParams *qp, O *out, cudaStream_t s) {
    const dim3 grid(flat_blocks((n + 15) / 16));
    switch (splits) {
    case 1: return launch(combine_kernel<O, 1>, grid, s, part, splits, n, qp, out);
    case 2: return launch(combine_kernel<O, 2>, grid, s, part, splits, n, qp, out);
    case 3: return launch(combine_kernel<O, 3>, grid, s, part, splits, n, qp, out);
    case 4: return launch(combine_kernel<O, 4>, grid, s, part, splits, n, qp, out);
    default: return launch(combine_kernel<O, 0>, dim3(flat_blocks(n)), s, part, splits, n, qp, out);
    }
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
    // the images split in groups so that about 16 blocks per SM run
    const int64_t pix_blocks = (g.H * g.W + kThreads - 1) / kThreads * rows_cap(g.C);
    int64_t groups = (static_cast<int64_t>(device_sm_count()) * 16 + pix_blocks - 1) / pix_blocks;
    groups = groups < 1 ? 1 : (groups > g.B ? g.B : (groups > 65535 ? 65535 : groups));
    const int imgs = static_cast<int>((g.B + groups - 1) / groups);
    const dim3 pix_grid(static_cast<unsigned>((g.H * g.W + kThreads - 1) / kThreads), rows_cap(g.C),
                        static_cast<unsigned>((g.B + imgs - 1) / imgs));
    if (e == cudaSuccess) {
        if (g.s == 1) e = launch(colmax_x_kernel<TX, 1>, pix_grid, s, x, g, imgs, act);
        else if (g.s == 2) e = launch(colmax_x_kernel<TX, 2>, pix_grid, s, x, g, imgs, act);
        else e = launch(colmax_x_kernel<TX, 0>, pix_grid, s, x, g, imgs, act);
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
        const char *unfold = std::getenv("BT_W8A8_UNFOLD");     // "gather" forces the direct gather
        QTile u;
        const int es = smooth ? static_cast<int>(sizeof(TX)) : 2;     // window of x, or of codes
        if ((unfold == nullptr || std::strcmp(unfold, "gather") != 0) && plan_qtile(g, es, u) &&
            qtile_smem(u, es, smooth != 0) <= 48 * 1024) {
            const dim3 grid(static_cast<unsigned>(g.B * u.nb * u.nwc * u.ncu));
            const size_t sm = qtile_smem(u, es, smooth != 0);
            e = smooth ? launch_pdl_smem(quant_tile_kernel<TX, true>, grid, dim3(kThreads), sm, s, x, g, u,
                                         static_cast<const float *>(scale), static_cast<const QParams *>(qp), qx)
                       : launch_pdl_smem(quant_tile_kernel<TX, false>, grid, dim3(kThreads), sm, s, x, g, u,
                                         static_cast<const float *>(scale), static_cast<const QParams *>(qp), qx);
        } else {
            const dim3 qgrid(static_cast<unsigned>((g.P + kQP - 1) / kQP), static_cast<unsigned>((g.C + kQC - 1) / kQC));
            e = smooth ? launch(quant_rows_kernel<TX, true>, qgrid, s, x, g, static_cast<const float *>(scale),
                                static_cast<const QParams *>(qp), qx)
                       : launch(quant_rows_kernel<TX, false>, qgrid, s, x, g, static_cast<const float *>(scale),
                                static_cast<const QParams *>(qp), qx);
        }
    }
    if (e == cudaSuccess)
        e = launch_tc_bf16_splitk(qw, g.Tp, qx, g.Tp, g.O, g.P, g.Tp, splits, 1.0f, part, err, s, g.Ho * g.Wo);
    if (e == cudaSuccess) {
        const int64_t n = g.B * g.O * g.Ho * g.Wo;
        e = out_t == BT_F32 ? launch_combine(static_cast<const float *>(part), splits, n, static_cast<const QParams *>(qp),
                                             static_cast<float *>(out), s)
                            : launch_combine(static_cast<const float *>(part), splits, n, static_cast<const QParams *>(qp),
                                             static_cast<__nv_bfloat16 *>(out), s);
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
