// Fused shift + sign + pack (the activation shift of
// BinaryConv2dCutlass.set_activation, the sign binarization of the native
// forward, and the bit-packing of w_pack / generate_quantized_weight).
//
// Both layouts work on groups of 8 consecutive elements (channels), which map
// to one output byte (bits), 4 bytes (E2M1) or 8 bytes (E4M3):
//   rows   [R, K] -> [R, row_bytes(K)]: a thread takes 4 groups of a row,
//          each one or two 16-byte loads, all issued before any is used.
//   nhwc   [B, C, H, W] -> [B, H, W, row_bytes(C)]: a thread takes 8 channel
//          planes x one 16-byte run of pixels and writes each pixel's group.
// Both are HBM streams: the input is read once and written 1/32 (bits),
// 1/8 (E2M1) or 1/4 (E4M3) of its fp32 size.
#include <mutex>

#include "bt_device.cuh"
#include "bt_internal.h"
#include "tc_ptx.cuh"

namespace bt {
namespace {

constexpr int kPackThreads = 256;
constexpr int kRowThreads = 128;
constexpr int kGroupsPerThread = 4;    // 8-element groups in flight per thread

// Output bytes produced from one group of 8 elements (channels).
template <int CODE> struct GroupOut;
template <> struct GroupOut<BT_CODE_BITS> { static constexpr int kBytes = 1; };
template <> struct GroupOut<BT_CODE_E4M3> { static constexpr int kBytes = 8; };
template <> struct GroupOut<BT_CODE_E2M1> { static constexpr int kBytes = 4; };

// Elements covered by one packed row of rb bytes.
template <int CODE> __host__ __device__ __forceinline__ int64_t padded_elems(int64_t rb) {
    return CODE == BT_CODE_BITS ? rb * 8 : (CODE == BT_CODE_E4M3 ? rb : rb * 2);
}

// Loads of one group of 8 elements: one 16-byte vector for 2-byte types,
// two for fp32.
template <typename T> struct Group {
    static constexpr int kVecs = 8 / Elem<T>::kPerVec;
    uint4 q[kVecs];
    __device__ __forceinline__ void load(const T *p) {
#pragma unroll
        for (int v = 0; v < kVecs; ++v) q[v] = ld_stream_v4(p + v * Elem<T>::kPerVec);
    }
    __device__ __forceinline__ void unpack(float (&f)[8]) const {
#pragma unroll
        for (int v = 0; v < kVecs; ++v) Elem<T>::unpack(q[v], f + v * Elem<T>::kPerVec);
    }
};

// Codes of 8 values from their "negative" mask (bit e set where value e
// binarizes to -1) and their valid mask (bit e clear past the end of the row:
// code 0). The fast path (valid == 0xFF) is a few integer operations.
__device__ __forceinline__ uint32_t spread_nibbles(uint32_t b) {   // bit e -> bit 4e
    b = (b | (b << 12)) & 0x000F000Fu;
    b = (b | (b << 6)) & 0x03030303u;
    b = (b | (b << 3)) & 0x11111111u;
    return b;
}
__device__ __forceinline__ uint32_t spread4_bytes(uint32_t x) {    // bits 0..3 -> 0, 8, 16, 24
    x = (x | (x << 14)) & 0x00030003u;                             // 0, 1, 16, 17
    x = (x | (x << 7)) & 0x01010101u;                              // 0, 8, 16, 24
    return x;
}
__device__ __forceinline__ uint64_t spread_bytes(uint32_t b) {     // bit e -> bit 8e
    return (static_cast<uint64_t>(spread4_bytes((b >> 4) & 0xFu)) << 32) | spread4_bytes(b & 0xFu);
}

template <int CODE>
__device__ __forceinline__ void store_group(uint8_t *dst, uint32_t neg, uint32_t valid) {
    if (CODE == BT_CODE_BITS) {
        *dst = static_cast<uint8_t>(~neg & valid);
    } else if (CODE == BT_CODE_E4M3) {
        // +1 = 0x38, -1 = 0xB8 (sign bit 7), padding 0x00
        const uint64_t n = spread_bytes(neg) << 7;
        uint64_t w = 0x3838383838383838ull | n;
        if (valid != 0xFFu) w &= spread_bytes(valid) * 0xFFull;
        *reinterpret_cast<uint2 *>(dst) = make_uint2(static_cast<uint32_t>(w), static_cast<uint32_t>(w >> 32));
    } else {
        // +1 = 0x2, -1 = 0xA (sign bit 3), padding 0x0
        uint32_t w = 0x22222222u | (spread_nibbles(neg) << 3);
        if (valid != 0xFFu) w &= spread_nibbles(valid) * 0xFu;
        *reinterpret_cast<uint32_t *>(dst) = w;
    }
}

// rows: one thread per group of 8 consecutive elements of a row, kGroupsPerThread
// groups (kRowThreads apart) per thread; blockIdx.y walks the rows. A group
// wholly inside the row is one or two 16-byte loads (VEC); the row's last,
// partial group and rows that are not 16-byte aligned take per-element loads.
template <typename T, int CODE, bool VEC>
__global__ void __launch_bounds__(kRowThreads)
pack_rows_kernel(const T *__restrict__ x, int64_t R, int K, const float *__restrict__ bias, int bias_len,
                 uint8_t *__restrict__ out, int rb, int G) {
    constexpr int OB = GroupOut<CODE>::kBytes;
    pdl_launch_dependents();
    pdl_wait();
    const float bs = bias_len == 1 ? __ldg(bias) : 0.0f;
    for (int64_t row = blockIdx.y; row < R; row += gridDim.y) {
        const T *xr = x + row * K;
        uint8_t *orow = out + row * rb;
        const int g0 = blockIdx.x * (kRowThreads * kGroupsPerThread) + threadIdx.x;

        Group<T> grp[kGroupsPerThread];
#pragma unroll
        for (int u = 0; u < kGroupsPerThread; ++u) {
            const int g = g0 + u * kRowThreads;
            if (VEC && g < G && 8 * g + 8 <= K) grp[u].load(xr + 8 * g);
        }
#pragma unroll
        for (int u = 0; u < kGroupsPerThread; ++u) {
            const int g = g0 + u * kRowThreads;
            if (g >= G) continue;
            const int k0 = 8 * g;
            float f[8];
            uint32_t valid = 0xFFu;
            if (VEC && k0 + 8 <= K) {
                grp[u].unpack(f);
            } else {
                valid = 0;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const bool in = k0 + e < K;
                    f[e] = in ? Elem<T>::to_f32(xr[k0 + e]) : 0.0f;
                    valid |= (in ? 1u : 0u) << e;
                }
            }
            uint32_t neg = 0;
            if (bias_len > 1) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float b = ((valid >> e) & 1u) ? __ldg(bias + k0 + e) : 0.0f;
                    neg |= is_negative(f[e], b) << e;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) neg |= is_negative(f[e], bs) << e;
            }
            store_group<CODE>(orow + static_cast<int64_t>(g) * OB, neg, valid);
        }
    }
}

// rows, staged: for 16-byte aligned rows. Each CTA walks "units" (a row, or a
// <= 16 KB segment of a long row); one thread keeps kStagedStages units in
// flight with bulk async copies into a shared-memory ring, and all threads
// convert the landed unit group by group (consecutive threads, consecutive
// 16-byte reads and consecutive output bytes). The unit that ends a row also
// writes the row's zero padding.
constexpr int kStagedThreads = 256;
constexpr int kStagedStages = 4;
constexpr int kSegBytes = 16384;
constexpr int kStagedSmem = kStagedStages * kSegBytes + 128;

template <typename T, int CODE>
__global__ void __launch_bounds__(kStagedThreads)
pack_rows_staged_kernel(const T *__restrict__ x, int64_t R, int K, const float *__restrict__ bias, int bias_len,
                        uint8_t *__restrict__ out, int rb, int G, int seg, int upr, unsigned int *err) {
    constexpr int OB = GroupOut<CODE>::kBytes;
    constexpr int S = kStagedStages;
    extern __shared__ __align__(128) uint8_t sm[];
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bars = sbase + S * kSegBytes;
    volatile uint32_t *flag = reinterpret_cast<volatile uint32_t *>(sm + S * kSegBytes + 8 * S);
    const int tid = threadIdx.x;
    const int64_t U = R * upr;
    const float bs = bias_len == 1 ? __ldg(bias) : 0.0f;
    const int data_groups = (K + 7) / 8;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) tc::mbar_init(bars + 8u * s, 1);
        *flag = 0u;
        tc::fence_mbar_init();
    }
    pdl_launch_dependents();
    __syncthreads();
    pdl_wait();

    auto issue = [&](int64_t unit, int s) {
        const int64_t row = unit / upr;
        const int k0 = static_cast<int>(unit - row * upr) * seg;
        const int len = K - k0 < seg ? K - k0 : seg;
        const uint32_t bytes = static_cast<uint32_t>(len) * sizeof(T);
        tc::mbar_arrive_expect_tx(bars + 8u * s, bytes);
        tc::bulk_load_once(sbase + s * kSegBytes, x + row * K + k0, bytes, bars + 8u * s);
    };
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            const int64_t unit = blockIdx.x + static_cast<int64_t>(s) * gridDim.x;
            if (unit < U) issue(unit, s);
        }
    }

    int i = 0;
    int64_t unit = blockIdx.x;
    for (; unit < U; unit += gridDim.x, ++i) {
        const int s = i % S;
        const uint32_t ph = static_cast<uint32_t>(i / S) & 1u;
        if (tid == 0) (void)tc::wait_bounded(bars + 8u * s, ph, flag, err);
        __syncthreads();
        if (*flag) break;
        (void)tc::mbar_try_wait(bars + 8u * s, ph);       // completed phase: acquire for this thread
        const int64_t row = unit / upr;
        const int k0 = static_cast<int>(unit - row * upr) * seg;
        const int len = K - k0 < seg ? K - k0 : seg;
        const T *sx = reinterpret_cast<const T *>(sm + s * kSegBytes);
        uint8_t *orow = out + row * rb;
        const int ngroups = (len + 7) / 8;
        for (int gl = tid; gl < ngroups; gl += kStagedThreads) {
            const int kl = 8 * gl;
            float f[8];
            uint32_t valid = 0xFFu;
            if (kl + 8 <= len) {
                Group<T> grp;
#pragma unroll
                for (int v = 0; v < Group<T>::kVecs; ++v)
                    grp.q[v] = *reinterpret_cast<const uint4 *>(sx + kl + v * Elem<T>::kPerVec);
                grp.unpack(f);
            } else {
                valid = 0;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const bool in = kl + e < len;
                    f[e] = in ? Elem<T>::to_f32(sx[kl + e]) : 0.0f;
                    valid |= (in ? 1u : 0u) << e;
                }
            }
            uint32_t neg = 0;
            if (bias_len > 1) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float b = ((valid >> e) & 1u) ? __ldg(bias + k0 + kl + e) : 0.0f;
                    neg |= is_negative(f[e], b) << e;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) neg |= is_negative(f[e], bs) << e;
            }
            store_group<CODE>(orow + static_cast<int64_t>(k0 / 8 + gl) * OB, neg, valid);
        }
        if (k0 + len == K) {
            for (int g = data_groups + tid; g < G; g += kStagedThreads)
                store_group<CODE>(orow + static_cast<int64_t>(g) * OB, 0u, 0u);
        }
        __syncthreads();
        if (tid == 0) {
            const int64_t next = unit + static_cast<int64_t>(S) * gridDim.x;
            if (next < U) {
                tc::fence_proxy_async_smem();
                issue(next, s);
            }
        }
    }
    if (tid == 0 && *flag) {
        // aborted: let the copies still in flight land before the CTA exits
        for (int k = 0; k < S; ++k, ++i, unit += gridDim.x) {
            if (unit >= U) break;
            const unsigned long long t0 = globaltimer_ns();
            while (!tc::mbar_try_wait(bars + 8u * (i % S), static_cast<uint32_t>(i / S) & 1u) &&
                   globaltimer_ns() - t0 < kWaitNs) {}
        }
    }
}

// nhwc: one thread per (image b, group of E consecutive pixels, group of 8
// channels); the 8 x E loads are 16 bytes each, consecutive threads taking
// consecutive pixel groups of the same channel planes. Each pixel gets the
// group's 1 (bits) / 4 (E2M1) / 8 (E4M3) output bytes.
template <typename T, int CODE, bool VEC>
__global__ void __launch_bounds__(kPackThreads)
pack_nhwc_kernel(const T *__restrict__ x, int B, int C, int HW, const float *__restrict__ bias, int bias_len,
                 uint8_t *__restrict__ out, int rb) {
    constexpr int E = Elem<T>::kPerVec;            // pixels per thread
    constexpr int OB = GroupOut<CODE>::kBytes;
    const uint32_t npg = static_cast<uint32_t>((HW + E - 1) / E);
    const uint32_t ncg = static_cast<uint32_t>(padded_elems<CODE>(rb) / 8);
    const uint64_t total = static_cast<uint64_t>(B) * ncg * npg;
    pdl_launch_dependents();
    pdl_wait();
    const float bs = bias_len == 1 ? __ldg(bias) : 0.0f;

    for (uint64_t t = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
         t += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
        const uint32_t pg = static_cast<uint32_t>(t % npg);
        const uint64_t rest = t / npg;
        const uint32_t cg = static_cast<uint32_t>(rest % ncg);
        const int64_t b = static_cast<int64_t>(rest / ncg);
        const int p0 = static_cast<int>(pg) * E;
        const int c0 = static_cast<int>(cg) * 8;

        float f[8][E];
        uint32_t cvalid = 0;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
            const int c = c0 + cc;
            if (c < C) {
                cvalid |= 1u << cc;
                const T *src = x + (b * C + c) * static_cast<int64_t>(HW) + p0;
                if (VEC) {
                    Elem<T>::unpack(ld_stream_v4(src), f[cc]);
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e) f[cc][e] = (p0 + e < HW) ? Elem<T>::to_f32(src[e]) : 0.0f;
                }
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) f[cc][e] = 0.0f;
            }
        }
        float bv[8];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
            bv[cc] = (bias_len > 1 && ((cvalid >> cc) & 1u)) ? __ldg(bias + c0 + cc) : bs;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            if (p0 + e >= HW) break;
            uint32_t neg = 0;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) neg |= is_negative(f[cc][e], bv[cc]) << cc;
            store_group<CODE>(out + ((b * HW + p0 + e) * static_cast<int64_t>(rb) + static_cast<int64_t>(cg) * OB),
                              neg, cvalid);
        }
    }
}

int grid_for(int64_t threads) {
    int64_t blocks = (threads + kPackThreads - 1) / kPackThreads;
    const int64_t cap = int64_t(1) << 30;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

template <typename T, int CODE>
cudaError_t rows_t(const T *x, int64_t R, int64_t K, const float *bias, int64_t bias_len, uint8_t *out,
                   int64_t rb, cudaStream_t s) {
    const int64_t G = padded_elems<CODE>(rb) / 8;
    const int64_t per_block = kRowThreads * kGroupsPerThread;
    dim3 grid(static_cast<unsigned>((G + per_block - 1) / per_block), static_cast<unsigned>(R < 65535 ? R : 65535));
    const bool vec = ((K * static_cast<int64_t>(sizeof(T))) % 16 == 0) && aligned(x, 16);
    unsigned int *err = device_error_word();
    if (vec && err != nullptr) {
        auto kern = pack_rows_staged_kernel<T, CODE>;
        static std::once_flag once;
        static cudaError_t attr = cudaSuccess;
        std::call_once(once, [&] {
            attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kStagedSmem);
        });
        if (attr != cudaSuccess) return attr;
        const int seg = kSegBytes / static_cast<int>(sizeof(T));
        const int64_t upr = (K + seg - 1) / seg;
        int sms = 0, dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int64_t units = R * upr;
        const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 148) * 3;
        const int grid = static_cast<int>(units < cap ? units : cap);
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute pdl = pdl_attribute();
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(kStagedThreads);
        cfg.dynamicSmemBytes = kStagedSmem;
        cfg.stream = s;
        cfg.attrs = &pdl;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, x, R, static_cast<int>(K), bias, static_cast<int>(bias_len), out,
                                  static_cast<int>(rb), static_cast<int>(G), seg, static_cast<int>(upr), err);
    }
    if (vec)
        pack_rows_kernel<T, CODE, true><<<grid, kRowThreads, 0, s>>>(x, R, static_cast<int>(K), bias,
                                                                     static_cast<int>(bias_len), out,
                                                                     static_cast<int>(rb), static_cast<int>(G));
    else
        pack_rows_kernel<T, CODE, false><<<grid, kRowThreads, 0, s>>>(x, R, static_cast<int>(K), bias,
                                                                      static_cast<int>(bias_len), out,
                                                                      static_cast<int>(rb), static_cast<int>(G));
    return cudaGetLastError();
}

template <typename T, int CODE>
cudaError_t nhwc_t(const T *x, int64_t B, int64_t C, int64_t HW, const float *bias, int64_t bias_len,
                   uint8_t *out, int64_t rb, cudaStream_t s) {
    constexpr int E = Elem<T>::kPerVec;
    const int64_t threads = B * (padded_elems<CODE>(rb) / 8) * ((HW + E - 1) / E);
    const int grid = grid_for(threads);
    const bool vec = ((HW * static_cast<int64_t>(sizeof(T))) % 16 == 0) && aligned(x, 16);
    if (vec)
        pack_nhwc_kernel<T, CODE, true><<<grid, kPackThreads, 0, s>>>(x, static_cast<int>(B), static_cast<int>(C),
                                                                      static_cast<int>(HW), bias,
                                                                      static_cast<int>(bias_len), out,
                                                                      static_cast<int>(rb));
    else
        pack_nhwc_kernel<T, CODE, false><<<grid, kPackThreads, 0, s>>>(x, static_cast<int>(B), static_cast<int>(C),
                                                                       static_cast<int>(HW), bias,
                                                                       static_cast<int>(bias_len), out,
                                                                       static_cast<int>(rb));
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
