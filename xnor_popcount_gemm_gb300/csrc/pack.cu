// Fused shift + sign + pack (the activation shift of
// BinaryConv2dCutlass.set_activation, the sign binarization of the native
// forward, and the bit-packing of w_pack / generate_quantized_weight).
//
// Two layouts:
//   rows   [R, K] -> [R, row_bytes(K)]: each warp walks 16-byte vector loads
//          along a row; lanes that cover one 32-bit word OR their bits
//          together with shuffles; codes are written as they are formed.
//   nhwc   [B, C, H, W] -> [B, H, W, row_bytes(C)]: each thread loads 16 bytes
//          of consecutive pixels from 16 or 32 channel planes (coalesced along
//          the pixels) and writes the packed channel group of each pixel.
// Both are pure HBM streams: read the input once, write 1/32 (bits), 1/8
// (E2M1) or 1/4 (E4M3) of an fp32 input's bytes.
#include "bt_device.cuh"
#include "bt_internal.h"

namespace bt {
namespace {

constexpr int kPackThreads = 256;
constexpr int kStepsPerChunk = 4;   // 16-byte loads in flight per lane

__device__ __forceinline__ float bias_at(const float *__restrict__ bias, int64_t bias_len, int64_t i) {
    if (bias_len == 0) return 0.0f;
    if (bias_len == 1) return __ldg(bias);
    return __ldg(bias + i);
}

template <typename T, int CODE, bool VEC>
__global__ void __launch_bounds__(kPackThreads)
pack_rows_kernel(const T *__restrict__ x, int64_t R, int64_t K, const float *__restrict__ bias,
                 int64_t bias_len, uint8_t *__restrict__ out, int64_t rb, int64_t steps_per_row,
                 int64_t chunks_per_row) {
    constexpr int E = Elem<T>::kPerVec;     // elements per lane per step
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t items = R * chunks_per_row;

    for (int64_t it = warp0; it < items; it += nwarps) {      // warp-uniform loop
        const int64_t row = it / chunks_per_row;
        const int64_t chunk = it - row * chunks_per_row;
        const T *xr = x + row * K;
        uint8_t *orow = out + row * rb;

        float f[kStepsPerChunk][E];
#pragma unroll
        for (int st = 0; st < kStepsPerChunk; ++st) {
            const int64_t step = chunk * kStepsPerChunk + st;
            const int64_t k0 = (step * 32 + lane) * E;
            if (VEC) {
                // K * sizeof(T) is a multiple of 16: a vector is wholly in or out.
                if (step < steps_per_row && k0 < K) {
                    Elem<T>::unpack(ld_stream_v4(xr + k0), f[st]);
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e) f[st][e] = 0.0f;
                }
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int64_t k = k0 + e;
                    f[st][e] = (step < steps_per_row && k < K) ? Elem<T>::to_f32(xr[k]) : 0.0f;
                }
            }
        }

#pragma unroll
        for (int st = 0; st < kStepsPerChunk; ++st) {
            const int64_t step = chunk * kStepsPerChunk + st;
            if (step >= steps_per_row) break;                  // warp-uniform
            const int64_t k0 = (step * 32 + lane) * E;
            uint32_t bits = 0, valid = 0;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int64_t k = k0 + e;
                if (k < K) {
                    bits |= sign_bit(f[st][e], bias_at(bias, bias_len, k)) << e;
                    valid |= 1u << e;
                }
            }
            if (CODE == BT_CODE_BITS) {
                constexpr int G = 32 / E;                      // lanes per 32-bit word
                uint32_t v = bits << ((lane % G) * E);
#pragma unroll
                for (int off = G / 2; off > 0; off >>= 1) v |= __shfl_xor_sync(0xffffffffu, v, off);
                const int64_t word = step * E + lane / G;
                if ((lane % G) == 0 && word * 4 < rb) reinterpret_cast<uint32_t *>(orow)[word] = v;
            } else if (CODE == BT_CODE_E4M3) {
                if (k0 < rb) {
                    uint32_t w[E / 4];
#pragma unroll
                    for (int q = 0; q < E / 4; ++q) {
                        w[q] = 0;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int idx = 4 * q + e;
                            const uint32_t c = ((valid >> idx) & 1u) ? e4m3_code((bits >> idx) & 1u) : 0u;
                            w[q] |= c << (8 * e);
                        }
                    }
                    if (E == 8) *reinterpret_cast<uint2 *>(orow + k0) = make_uint2(w[0], w[E / 4 - 1]);
                    else *reinterpret_cast<uint32_t *>(orow + k0) = w[0];
                }
            } else {   // E2M1: E nibbles = E/2 bytes at byte k0/2
                if (k0 / 2 < rb) {
                    uint32_t w = 0;
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const uint32_t c = ((valid >> e) & 1u) ? e2m1_code((bits >> e) & 1u) : 0u;
                        w |= c << (4 * e);
                    }
                    if (E == 8) *reinterpret_cast<uint32_t *>(orow + k0 / 2) = w;
                    else *reinterpret_cast<uint16_t *>(orow + k0 / 2) = static_cast<uint16_t>(w);
                }
            }
        }
    }
}

template <typename T, int CODE, bool VEC>
__global__ void __launch_bounds__(kPackThreads)
pack_nhwc_kernel(const T *__restrict__ x, int64_t B, int64_t C, int64_t HW,
                 const float *__restrict__ bias, int64_t bias_len, uint8_t *__restrict__ out,
                 int64_t rb) {
    constexpr int E = Elem<T>::kPerVec;                        // pixels per thread
    constexpr int CG = (CODE == BT_CODE_E4M3) ? 16 : 32;       // channels per thread
    constexpr int GB = (CODE == BT_CODE_BITS) ? 4 : 16;        // output bytes per pixel
    constexpr int GW = GB / 4;
    const int64_t npg = (HW + E - 1) / E;
    const int64_t ncg = rb / GB;
    const int64_t total = B * ncg * npg;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;

    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total; t += stride) {
        const int64_t pg = t % npg;
        const int64_t rest = t / npg;
        const int64_t cg = rest % ncg;
        const int64_t b = rest / ncg;
        const int64_t p0 = pg * E;

        uint32_t acc[E][GW];
#pragma unroll
        for (int e = 0; e < E; ++e)
#pragma unroll
            for (int q = 0; q < GW; ++q) acc[e][q] = 0;

#pragma unroll
        for (int cc = 0; cc < CG; ++cc) {
            const int64_t c = cg * CG + cc;
            if (c < C) {
                const T *src = x + (b * C + c) * HW + p0;
                float f[E];
                if (VEC) {
                    Elem<T>::unpack(ld_stream_v4(src), f);
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e) f[e] = (p0 + e < HW) ? Elem<T>::to_f32(src[e]) : 0.0f;
                }
                const float bv = bias_at(bias, bias_len, c);
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const uint32_t bit = sign_bit(f[e], bv);
                    if (CODE == BT_CODE_BITS) acc[e][0] |= bit << cc;
                    else if (CODE == BT_CODE_E4M3) acc[e][cc / 4] |= e4m3_code(bit) << (8 * (cc % 4));
                    else acc[e][cc / 8] |= e2m1_code(bit) << (4 * (cc % 8));
                }
            }
        }
#pragma unroll
        for (int e = 0; e < E; ++e) {
            if (p0 + e < HW) {
                uint8_t *dst = out + ((b * HW + p0 + e) * rb + cg * GB);
                if (GW == 1) *reinterpret_cast<uint32_t *>(dst) = acc[e][0];
                else *reinterpret_cast<uint4 *>(dst) = make_uint4(acc[e][0], acc[e][GW > 1 ? 1 : 0],
                                                                  acc[e][GW > 2 ? 2 : 0], acc[e][GW > 3 ? 3 : 0]);
            }
        }
    }
}

int grid_for(int64_t threads) {
    int64_t blocks = (threads + kPackThreads - 1) / kPackThreads;
    const int64_t cap = 152 * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

template <typename T, int CODE>
cudaError_t rows_t(const T *x, int64_t R, int64_t K, const float *bias, int64_t bias_len, uint8_t *out,
                   int64_t rb, cudaStream_t s) {
    constexpr int E = Elem<T>::kPerVec;
    const int64_t padded = (CODE == BT_CODE_BITS) ? rb * 8 : (CODE == BT_CODE_E4M3 ? rb : rb * 2);
    const int64_t steps = (padded + 32 * E - 1) / (32 * E);
    const int64_t chunks = (steps + kStepsPerChunk - 1) / kStepsPerChunk;
    const int grid = grid_for(R * chunks * 32);
    const bool vec = ((K * static_cast<int64_t>(sizeof(T))) % 16 == 0) && aligned(x, 16);
    if (vec)
        pack_rows_kernel<T, CODE, true><<<grid, kPackThreads, 0, s>>>(x, R, K, bias, bias_len, out, rb, steps, chunks);
    else
        pack_rows_kernel<T, CODE, false><<<grid, kPackThreads, 0, s>>>(x, R, K, bias, bias_len, out, rb, steps, chunks);
    return cudaGetLastError();
}

template <typename T, int CODE>
cudaError_t nhwc_t(const T *x, int64_t B, int64_t C, int64_t HW, const float *bias, int64_t bias_len,
                   uint8_t *out, int64_t rb, cudaStream_t s) {
    constexpr int E = Elem<T>::kPerVec;
    constexpr int GB = (CODE == BT_CODE_BITS) ? 4 : 16;
    const int64_t threads = B * (rb / GB) * ((HW + E - 1) / E);
    const int grid = grid_for(threads);
    const bool vec = ((HW * static_cast<int64_t>(sizeof(T))) % 16 == 0) && aligned(x, 16);
    if (vec)
        pack_nhwc_kernel<T, CODE, true><<<grid, kPackThreads, 0, s>>>(x, B, C, HW, bias, bias_len, out, rb);
    else
        pack_nhwc_kernel<T, CODE, false><<<grid, kPackThreads, 0, s>>>(x, B, C, HW, bias, bias_len, out, rb);
    return cudaGetLastError();
}

template <typename T>
cudaError_t rows_code(const T *x, int64_t R, int64_t K, const float *bias, int64_t bias_len, bt_code code,
                      void *out, cudaStream_t s) {
    uint8_t *o = static_cast<uint8_t *>(out);
    const int64_t rb = row_bytes(K, code);
    switch (code) {
        case BT_CODE_BITS: return rows_t<T, BT_CODE_BITS>(x, R, K, bias, bias_len, o, rb, s);
        case BT_CODE_E4M3: return rows_t<T, BT_CODE_E4M3>(x, R, K, bias, bias_len, o, rb, s);
        default: return rows_t<T, BT_CODE_E2M1>(x, R, K, bias, bias_len, o, rb, s);
    }
}

template <typename T>
cudaError_t nhwc_code(const T *x, int64_t B, int64_t C, int64_t HW, const float *bias, int64_t bias_len,
                      bt_code code, void *out, cudaStream_t s) {
    uint8_t *o = static_cast<uint8_t *>(out);
    const int64_t rb = row_bytes(C, code);
    switch (code) {
        case BT_CODE_BITS: return nhwc_t<T, BT_CODE_BITS>(x, B, C, HW, bias, bias_len, o, rb, s);
        case BT_CODE_E4M3: return nhwc_t<T, BT_CODE_E4M3>(x, B, C, HW, bias, bias_len, o, rb, s);
        default: return nhwc_t<T, BT_CODE_E2M1>(x, B, C, HW, bias, bias_len, o, rb, s);
    }
}

}  // namespace

cudaError_t launch_pack_rows(const void *x, bt_dtype xt, int64_t R, int64_t K, const float *bias,
                             int64_t bias_len, bt_code code, void *out, cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    switch (xt) {
        case BT_F32: return rows_code(static_cast<const float *>(x), R, K, bias, bias_len, code, out, s);
        case BT_BF16: return rows_code(static_cast<const __nv_bfloat16 *>(x), R, K, bias, bias_len, code, out, s);
        default: return rows_code(static_cast<const __half *>(x), R, K, bias, bias_len, code, out, s);
    }
}

cudaError_t launch_pack_nhwc(const void *x, bt_dtype xt, int64_t B, int64_t C, int64_t HW,
                             const float *bias, int64_t bias_len, bt_code code, void *out,
                             cudaStream_t s) {
    if (B == 0) return cudaSuccess;
    switch (xt) {
        case BT_F32: return nhwc_code(static_cast<const float *>(x), B, C, HW, bias, bias_len, code, out, s);
        case BT_BF16: return nhwc_code(static_cast<const __nv_bfloat16 *>(x), B, C, HW, bias, bias_len, code, out, s);
        default: return nhwc_code(static_cast<const __half *>(x), B, C, HW, bias, bias_len, code, out, s);
    }
}

}  // namespace bt
