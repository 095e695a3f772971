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
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "bt_device.cuh"
#include "bt_internal.h"
#include "sign_pack.cuh"
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

// Codes of a full group of 8 from its masks.
template <int CODE>
__device__ __forceinline__ void store_masks(uint8_t *dst, uint32_t P0, uint32_t P1) {
    if (CODE == BT_CODE_BITS) {
        *dst = static_cast<uint8_t>(mask_byte(P0, P1));
    } else if (CODE == BT_CODE_E4M3) {
        // +1 = 0x38, -1 = 0xB8
        *reinterpret_cast<uint2 *>(dst) = make_uint2(0x38383838u | (~P0 & 0x80808080u), 0x38383838u | (~P1 & 0x80808080u));
    } else {
        // +1 = 0x2, -1 = 0xA; value 2i in the low nibble of byte i
        const uint32_t even = __byte_perm(P0, P1, 0x6420), odd = __byte_perm(P0, P1, 0x7531);
        *reinterpret_cast<uint32_t *>(dst) = 0x22222222u | (~even & 0x08080808u) | (~odd & 0x80808080u);
    }
}

// Sum of |x| for the first-call activation scale, kept per thread as a
// compensated fp32 pair (Neumaier: s + c), then added in double across the
// warp and once per warp to the accumulator. An infinite term leaves the sum
// infinite (no compensation of inf - inf).
struct AbsSum {
    float s = 0.0f, c = 0.0f;
    __device__ __forceinline__ void add(float v) {
        const float t = s + v;
        if (isfinite(t)) c += fabsf(s) >= fabsf(v) ? (s - t) + v : (v - t) + s;
        s = t;
    }
    template <typename T> __device__ __forceinline__ void add_group(const Group<T> &g) {
        float f[8];
        g.unpack(f);
        add(((fabsf(f[0]) + fabsf(f[1])) + (fabsf(f[2]) + fabsf(f[3]))) +
            ((fabsf(f[4]) + fabsf(f[5])) + (fabsf(f[6]) + fabsf(f[7]))));
    }
    // every lane of the warp calls it
    __device__ __forceinline__ void flush(double *acc) {
        double d = static_cast<double>(s) + static_cast<double>(c);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xFFFFFFFFu, d, o);
        if ((threadIdx.x & 31) == 0) atomicAdd(acc, d);
    }
};

// rows, flat: every output group of every row, numbered g = row * G + j over
// the whole [R, G] output, kFlatUnroll per thread in flight. Group j < Gf
// holds elements 8j..8j+7 of the row and is read with VB-byte vectors (rows
// VB-aligned); a last, partial group (K not a multiple of 8) is read element
// by element; groups from Gd = ceil(K / 8) on are the row's zero padding.
// Consecutive threads take consecutive groups: contiguous loads and stores.
constexpr int kFlatUnroll = 4;

template <typename T, int CODE, bool COLBIAS, int VB, bool SUM = false>
__global__ void __launch_bounds__(kPackThreads)
pack_rows_flat_kernel(const T *__restrict__ x, uint32_t total, FastDiv divG, uint32_t Gf, int K,
                      const float *__restrict__ bias, int bias_len, uint8_t *__restrict__ out,
                      double *__restrict__ abs_sum = nullptr) {
    constexpr int OB = GroupOut<CODE>::kBytes;
    AbsSum asum;
    pdl_launch_dependents();
    pdl_wait();
    const float bs = bias_len == 1 ? __ldg(bias) : 0.0f;
    const bool finite = isfinite(bs);
    const uint32_t Gd = static_cast<uint32_t>((K + 7) / 8);
    const uint32_t stride = gridDim.x * (kPackThreads * kFlatUnroll);
    for (uint32_t g0 = blockIdx.x * (kPackThreads * kFlatUnroll) + threadIdx.x; g0 < total; g0 += stride) {
        Group<T> grp[kFlatUnroll];
        uint32_t col[kFlatUnroll], row[kFlatUnroll];
#pragma unroll
        for (int u = 0; u < kFlatUnroll; ++u) {
            const uint32_t g = g0 + u * kPackThreads;
            row[u] = fdiv(g, divG);
            col[u] = g - row[u] * divG.d;
            if (g < total && col[u] < Gf) grp[u].template load<VB>(x + static_cast<int64_t>(row[u]) * K + 8 * col[u]);
        }
#pragma unroll
        for (int u = 0; u < kFlatUnroll; ++u) {
            const uint32_t g = g0 + u * kPackThreads;
            if (g >= total) break;
            uint8_t *dst = out + static_cast<int64_t>(g) * OB;
            if (col[u] >= Gf) {
                uint32_t neg = 0, valid = 0;
                if (col[u] < Gd) {
                    // the row's last, partial group
                    const int k0 = 8 * static_cast<int>(col[u]);
                    const T *xr = x + static_cast<int64_t>(row[u]) * K;
                    for (int e = 0; e < K - k0; ++e) {
                        const float b = COLBIAS ? __ldg(bias + k0 + e) : bs;
                        const float v = Elem<T>::to_f32(xr[k0 + e]);
                        neg |= is_negative(v, b) << e;
                        valid |= 1u << e;
                        if constexpr (SUM) asum.add(fabsf(v));
                    }
                }
                store_group<CODE>(dst, neg, valid);             // (or row padding: code 0)
                continue;
            }
            if constexpr (SUM) asum.add_group(grp[u]);
            uint32_t P0, P1;
            if (!COLBIAS && finite) {
                masks_ge<T>(grp[u], -bs, P0, P1);
            } else {
                float f[8], b[8];
                grp[u].unpack(f);
                if (COLBIAS) {
                    const float4 b0 = __ldg(reinterpret_cast<const float4 *>(bias + 8 * col[u]));
                    const float4 b1 = __ldg(reinterpret_cast<const float4 *>(bias + 8 * col[u] + 4));
                    b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
                    b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) b[e] = bs;
                }
                masks_add(f, b, P0, P1);
            }
            store_masks<CODE>(dst, P0, P1);
        }
    }
    if constexpr (SUM) asum.flush(abs_sum);
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
                grp.load_smem(sx + kl);
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
    pdl_wait();
    // dependents start only after this wait: a convolution that follows may read its
    // weights before its own wait, and those may come from the kernel before this one
    pdl_launch_dependents();
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

// Transpose of an 8 x 8 bit matrix held as 8 bytes (byte i = row i, bit j =
// column j) into byte j = column j, bit i = row i: three rounds of swapping
// blocks across the diagonal (the transpose8 method of Warren, Hacker's
// Delight, section 7-3).
__device__ __forceinline__ uint64_t transpose8x8(uint64_t v) {
    uint64_t t = (v ^ (v >> 7)) & 0x00AA00AA00AA00AAull;
    v = v ^ t ^ (t << 7);
    t = (v ^ (v >> 14)) & 0x0000CCCC0000CCCCull;
    v = v ^ t ^ (t << 14);
    t = (v ^ (v >> 28)) & 0x00000000F0F0F0F0ull;
    return v ^ t ^ (t << 28);
}

// nhwc, warp-level. A unit is (image b, 32 consecutive pixels, 32 channels)
// and belongs to one warp. Loads: in round k (0..3) lane l reads 8 pixels
// (one 16-byte load for a 2-byte type, two for f32) of channel 8k + l / 4,
// pixels 8 (l % 4) .. + 7, so each load instruction covers 8 channel planes
// with 64 (128) contiguous bytes each, and turns them into one byte of sign
// bits (bit = +1). Lane l's word then holds bit (c, p) for channel c = 8k +
// (l >> 2) and pixel p = 8 (l & 3) + b at register bit 8k + b: lane bits
// (c2 c1 c0 p4 p3), register bits (c4 c3 p2 p1 p0). Three rounds of shuffles
// exchange lane bits 4, 3, 2 with register bits 2, 1, 0 (the off-diagonal
// blocks of a bit-matrix transpose), and one shuffle permutes the lanes to
// (p4 p3 p2 p1 p0): lane p ends with the word of pixel p, bit c for channel c.
// It turns that into codes and stores them (4 bytes of bits, 16 of E2M1, 32
// of E4M3) at its place in the pixel's packed row. No shared memory, no block
// barrier. Consecutive warps take consecutive pixel blocks of the same
// channels. Channels past C are code 0 (the row's zero padding). Needs every
// channel plane 16-byte aligned and HW a multiple of 4 (f32) or 8 (2-byte
// types); pixels past HW are neither loaded nor stored. (Measured on GB300
// inside a convolution step, this layout beat both the shared-memory
// transpose and a variant with one 512-byte plane run per load instruction.)
template <int CODE> struct Group32;
template <> struct Group32<BT_CODE_BITS> { static constexpr int kBytes = 4; };
template <> struct Group32<BT_CODE_E2M1> { static constexpr int kBytes = 16; };
template <> struct Group32<BT_CODE_E4M3> { static constexpr int kBytes = 32; };
constexpr int kWarpPackPixels = 32;

template <typename T, int CODE, bool SUM = false>
__global__ void __launch_bounds__(kPackThreads)
pack_nhwc_warp_kernel(const T *__restrict__ x, int C, int HW, uint32_t units, FastDiv div_npb, FastDiv div_ncg,
                      const float *__restrict__ bias, int bias_len, uint8_t *__restrict__ out, int rb,
                      double *__restrict__ abs_sum = nullptr) {
    constexpr int OB = Group32<CODE>::kBytes;
    AbsSum asum;
    const int lane = threadIdx.x & 31;
    const uint32_t warp0 = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
    const int ncg = static_cast<int>(div_ncg.d), npb = static_cast<int>(div_npb.d);
    const int j = lane & 3;                                // this lane's 8-pixel chunk in the loads
    pdl_wait();
    // dependents start only after this wait: a convolution that follows may read its
    // weights before its own wait, and those may come from the kernel before this one
    pdl_launch_dependents();
    const float bs = bias_len == 1 ? __ldg(bias) : 0.0f;
    for (uint32_t u = warp0; u < units; u += nwarps) {
        const uint32_t rest = fdiv(u, div_npb);
        const int p0 = static_cast<int>(u - rest * static_cast<uint32_t>(npb)) * kWarpPackPixels;
        const uint32_t bimg = fdiv(rest, div_ncg);
        const int cg = static_cast<int>(rest - bimg * static_cast<uint32_t>(ncg));
        const int64_t b = bimg;
        const int px = p0 + 8 * j;
        const int nvalid_px = HW - px;                     // pixels of this lane's chunk inside the image
        // all four rounds' loads go out before any of them is used
        Group<T> g[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int c = cg * 32 + 8 * k + (lane >> 2);
#pragma unroll
            for (int i = 0; i < Group<T>::kWords; ++i) g[k].w[i] = 0u;
            if (c < C && nvalid_px > 0) {
                const uint4 *src = reinterpret_cast<const uint4 *>(x + (b * C + c) * static_cast<int64_t>(HW) + px);
#pragma unroll
                for (int i = 0; i < Group<T>::kWords / 4; ++i) {
                    if (i == 0 || nvalid_px >= 8) {           // f32: the second half only if inside
                        const uint4 q = __ldg(src + i);
                        g[k].w[4 * i] = q.x; g[k].w[4 * i + 1] = q.y; g[k].w[4 * i + 2] = q.z; g[k].w[4 * i + 3] = q.w;
                    }
                }
            }
        }
        uint32_t w = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int c = cg * 32 + 8 * k + (lane >> 2);
            if (c < C && nvalid_px > 0) {
                if constexpr (SUM) asum.add_group(g[k]);         // zeros past HW add nothing
                const float bc = bias_len > 1 ? __ldg(bias + c) : bs;
                uint32_t P0, P1;
                if (isfinite(bc)) {
                    masks_ge<T>(g[k], -bc, P0, P1);
                } else {
                    float f[8], bb[8];
                    g[k].unpack(f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) bb[e] = bc;
                    masks_add(f, bb, P0, P1);
                }
                w |= mask_byte(P0, P1) << (8 * k);
            }
        }
        w = exchange_bits<16, 4, 0x0F0F0F0Fu>(w, lane);
        w = exchange_bits<8, 2, 0x33333333u>(w, lane);
        w = exchange_bits<4, 1, 0x55555555u>(w, lane);
        w = __shfl_sync(0xFFFFFFFFu, w, ((lane & 7) << 2) | (lane >> 3));
        // lane p: bit c = channel 32 cg + c at pixel p0 + p
        if (p0 + lane >= HW) continue;
        const int nvalid = C - cg * 32 >= 32 ? 32 : (C - cg * 32 > 0 ? C - cg * 32 : 0);
        const uint32_t valid = nvalid == 32 ? 0xFFFFFFFFu : (1u << nvalid) - 1u;
        uint8_t *dst = out + (b * HW + p0 + lane) * static_cast<int64_t>(rb) + cg * OB;
        const uint32_t neg = ~w & valid;
        if constexpr (CODE == BT_CODE_BITS) {
            *reinterpret_cast<uint32_t *>(dst) = w & valid;
        } else if constexpr (CODE == BT_CODE_E2M1) {
            uint32_t q[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t nb = (neg >> (8 * i)) & 0xFFu, vb = (valid >> (8 * i)) & 0xFFu;
                q[i] = 0x22222222u | (spread_nibbles(nb) << 3);
                if (vb != 0xFFu) q[i] &= spread_nibbles(vb) * 0xFu;
            }
            *reinterpret_cast<uint4 *>(dst) = make_uint4(q[0], q[1], q[2], q[3]);
        } else {
            uint32_t q[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t nb = (neg >> (8 * i)) & 0xFFu, vb = (valid >> (8 * i)) & 0xFFu;
                uint64_t v = 0x3838383838383838ull | (spread_bytes(nb) << 7);
                if (vb != 0xFFu) v &= spread_bytes(vb) * 0xFFull;
                q[2 * i] = static_cast<uint32_t>(v);
                q[2 * i + 1] = static_cast<uint32_t>(v >> 32);
            }
            *reinterpret_cast<uint4 *>(dst) = make_uint4(q[0], q[1], q[2], q[3]);
            *reinterpret_cast<uint4 *>(dst + 16) = make_uint4(q[4], q[5], q[6], q[7]);
        }
    }
    if constexpr (SUM) asum.flush(abs_sum);
}

// nhwc, warp-level, E2M1 codes: the same units (32 channels x 32 pixels of
// one image per warp), converted the way the convolution's packing warps
// convert them. Lane l loads 8 pixels (16 bytes of a 2-byte type, 32 of f32)
// of channel 32 cg + 8 k + l / 4 as predicated loads (zeros past C or HW); the
// sign test x >= t is one comparison per pair of values (t the shift's
// threshold, per channel or one for all), its bits land at lane bits (c2 c1
// c0 p4 p3) and register bits (p0 p2 p1 c4 c3); three exchange rounds and one
// shuffle leave lane p with channel c at bit 4 (c % 8) + c / 8, so the codes
// of channels 8i..8i+7 are one shift and one logic op. Units are numbered with
// the pixel block fastest (the input, 8 to 16 times the output's bytes, is
// read in runs); each warp loads its next unit before it converts the
// current one.
template <typename T, bool CHAN>
__global__ void __launch_bounds__(kPackThreads)
pack_nhwc_e2m1_kernel(const T *__restrict__ x, int C, int HW, uint32_t units, FastDiv div_ncg, FastDiv div_npb,
                      const float *__restrict__ bias, int bias_len, uint8_t *__restrict__ out, int rb) {
    constexpr int NV = sizeof(T) == 2 ? 1 : 2;                  // 16-byte loads per 8 pixels
    const int lane = threadIdx.x & 31;
    const uint32_t warp0 = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
    const int ncg = static_cast<int>(div_ncg.d), npb = static_cast<int>(div_npb.d);
    const int lc = lane >> 2, lp = 8 * (lane & 3);
    const int64_t hw8 = static_cast<int64_t>(8) * HW;
    const uint32_t keep16 = (lane & 16) ? 0xFFFF0000u : 0x0000FFFFu;
    const uint32_t keep8 = (lane & 8) ? 0xFF00FF00u : 0x00FF00FFu, rot8 = (lane & 8) ? 8u : 24u;
    const uint32_t keep4 = (lane & 4) ? 0xF0F0F0F0u : 0x0F0F0F0Fu, rot4 = (lane & 4) ? 4u : 28u;
    const int src_lane = ((lane & 1) << 4) | (((lane >> 2) & 1) << 3) | (((lane >> 1) & 1) << 2) |
                         (((lane >> 4) & 1) << 1) | ((lane >> 3) & 1);
    pdl_wait();
    // dependents start only after this wait: a convolution that follows may read its
    // weights before its own wait, and those may come from the kernel before this one
    pdl_launch_dependents();
    const uint32_t t_all = shift_threshold<T>(bias_len == 1 ? __ldg(bias) : 0.0f);
    // unit u: pixel block blk (fastest), then channel group cg of image b, so the
    // warps that run at the same time read long runs of the same channel planes
    auto decode = [&](uint32_t u, int &cg, int &b, int &blk) {
        const uint32_t q = fdiv(u, div_npb);
        blk = static_cast<int>(u - q * static_cast<uint32_t>(npb));
        const uint32_t bi = fdiv(q, div_ncg);
        cg = static_cast<int>(q - bi * static_cast<uint32_t>(ncg));
        b = static_cast<int>(bi);
    };
    auto load = [&](uint4 (&g)[4][NV], uint32_t u) {
        int cg, b, blk;
        decode(u, cg, b, blk);
        const int px = 32 * blk + lp;
        const int lim = C - cg * 32 - lc;
        const T *base = x + (static_cast<int64_t>(b) * C + cg * 32 + lc) * HW + px;
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int v = 0; v < NV; ++v)
                g[k][v] = ld_nc_v4_if(base + k * hw8 + 4 * v, 8 * k < lim && px + 4 * v < HW);
    };
    auto convert = [&](const uint4 (&g)[4][NV], uint32_t u) {
        int cg, b, blk;
        decode(u, cg, b, blk);
        uint32_t w = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t tk = t_all;
            if constexpr (CHAN) {
                const int c = cg * 32 + 8 * k + lc;
                tk = shift_threshold<T>(c < C ? __ldg(bias + c) : 0.0f);
            }
            w |= sign_bits<T>(g[k][0], g[k][NV - 1], tk, k);
        }
        w = exchange_rot(w, 16, keep16, 16u);
        w = exchange_rot(w, 8, keep8, rot8);
        w = exchange_rot(w, 4, keep4, rot4);
        w = __shfl_sync(0xFFFFFFFFu, w, src_lane);
        const int p = 32 * blk + lane;
        if (p >= HW) return;
        uint32_t q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = ((~w << (3 - i)) & 0x88888888u) | 0x22222222u;
        const int nvalid = C - cg * 32;
        if (nvalid < 32) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int nv = nvalid - 8 * i;            // channels of this word inside C
                if (nv < 8) q[i] &= nv <= 0 ? 0u : (1u << (4 * nv)) - 1u;
            }
        }
        *reinterpret_cast<uint4 *>(out + (static_cast<int64_t>(b) * HW + p) * rb + cg * 16) = make_uint4(q[0], q[1], q[2], q[3]);
    };
    uint4 g0[4][NV], g1[4][NV];
    uint32_t u = warp0;
    if (u < units) load(g0, u);
    while (u < units) {
        const uint32_t u1 = u + nwarps;
        if (u1 < units) load(g1, u1);
        convert(g0, u);
        u = u1;
        if (u >= units) break;
        const uint32_t u2 = u + nwarps;
        if (u2 < units) load(g0, u2);
        convert(g1, u);
        u = u2;
    }
}

// nhwc, transposed through shared memory. A unit is (image b, a run of
// kNhwcPixels pixels, every channel). Phase 1 reads each channel plane's run
// with 16-byte loads (consecutive threads, consecutive 8-pixel groups of a
// plane) and keeps one byte of sign bits per (pixel group, channel). Phase 2
// turns each 8 pixel x 8 channel block around with a bit-matrix transpose and
// writes the codes of whole pixel rows: consecutive threads take consecutive
// channel groups of a row, so every store instruction covers whole rows.
constexpr int kNhwcPixels = 64;
constexpr int kNhwcGroups = kNhwcPixels / 8;
constexpr int kNhwcUnroll = 4;
constexpr int kNhwcMaxSmem = 48 * 1024;

// Bytes of one pixel group's row of channel bytes in shared memory: the
// channels rounded up to 8, plus 8 so that consecutive rows start in
// different banks.
__host__ __device__ __forceinline__ int nhwc_cstride(int C) { return (C + 7) / 8 * 8 + 8; }

template <typename T, int CODE, bool VEC>
__global__ void __launch_bounds__(kPackThreads)
pack_nhwc_tr_kernel(const T *__restrict__ x, int C, int HW, int upi, uint32_t units, const float *__restrict__ bias,
                    int bias_len, uint8_t *__restrict__ out, int rb, FastDiv divG) {
    constexpr int OB = GroupOut<CODE>::kBytes;
    extern __shared__ __align__(16) uint8_t sbits[];      // [kNhwcGroups][cstride]
    const int cstride = nhwc_cstride(C);
    const int G = static_cast<int>(divG.d);
    const int tid = threadIdx.x;
    pdl_wait();
    // dependents start only after this wait: a convolution that follows may read its
    // weights before its own wait, and those may come from the kernel before this one
    pdl_launch_dependents();
    const float bs = bias_len == 1 ? __ldg(bias) : 0.0f;
    const int items1 = C * kNhwcGroups;

    for (uint32_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
        const int64_t b = unit / static_cast<uint32_t>(upi);
        const int p0 = static_cast<int>(unit - static_cast<uint32_t>(b) * upi) * kNhwcPixels;
        const int npx = HW - p0 < kNhwcPixels ? HW - p0 : kNhwcPixels;
        const T *xb = x + b * C * static_cast<int64_t>(HW) + p0;

        // phase 1: item it = (channel it / 8, pixel group it % 8)
        for (int base = 0; base < items1; base += kPackThreads * kNhwcUnroll) {
            Group<T> grp[kNhwcUnroll];
#pragma unroll
            for (int u = 0; u < kNhwcUnroll; ++u) {
                const int it = base + u * kPackThreads + tid;
                const int c = it >> 3, px = (it & 7) * 8;
                if (VEC && it < items1 && px + 8 <= npx) grp[u].load(xb + static_cast<int64_t>(c) * HW + px);
            }
#pragma unroll
            for (int u = 0; u < kNhwcUnroll; ++u) {
                const int it = base + u * kPackThreads + tid;
                if (it >= items1) break;
                const int c = it >> 3, pg = it & 7, px = pg * 8;
                if (px >= npx) continue;
                const float bc = bias_len > 1 ? __ldg(bias + c) : bs;
                const bool full = VEC && px + 8 <= npx;
                uint32_t P0, P1;
                if (full && isfinite(bc)) {
                    masks_ge<T>(grp[u], -bc, P0, P1);
                } else {
                    float f[8], bb[8];
                    if (full) {
                        grp[u].unpack(f);
                    } else {
                        const T *src = xb + static_cast<int64_t>(c) * HW + px;
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = px + e < npx ? Elem<T>::to_f32(src[e]) : 0.0f;
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) bb[e] = bc;
                    masks_add(f, bb, P0, P1);
                }
                sbits[pg * cstride + c] = static_cast<uint8_t>(mask_byte(P0, P1));
            }
        }
        __syncthreads();

        // phase 2: item it = (pixel group it / G, channel group it % G)
        const int npg = (npx + 7) >> 3;
        for (int it = tid; it < npg * G; it += kPackThreads) {
            const int pg = static_cast<int>(fdiv(static_cast<uint32_t>(it), divG));
            const int cg = it - pg * G;
            const int c0 = cg * 8;
            const int nj = npx - pg * 8 < 8 ? npx - pg * 8 : 8;
            uint8_t *dst = out + (b * HW + p0 + pg * 8) * static_cast<int64_t>(rb) + cg * OB;
            if (c0 >= C) {
                for (int j = 0; j < nj; ++j) store_group<CODE>(dst + static_cast<int64_t>(j) * rb, 0u, 0u);
                continue;
            }
            const uint32_t cvalid = C - c0 >= 8 ? 0xFFu : (1u << (C - c0)) - 1u;
            const uint64_t v = transpose8x8(*reinterpret_cast<const uint64_t *>(sbits + pg * cstride + c0));
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (j >= nj) break;
                const uint32_t pos = static_cast<uint32_t>(v >> (8 * j)) & 0xFFu;
                store_group<CODE>(dst + static_cast<int64_t>(j) * rb, ~pos & cvalid, cvalid);
            }
        }
        __syncthreads();
    }
}

// im2col rows (the unfold of the im2col write-up, on packed pixels): one
// thread per (output row m, 16-byte chunk c of a packed pixel) walks the k*k
// taps, so consecutive threads write consecutive chunks of a tap's slot in the
// row. The packed input is small and was just written (its reads hit L2); the
// rows are stored with plain stores so that they stay in L2 for the
// contraction that reads them next.
template <typename Idx>
__global__ void __launch_bounds__(kPackThreads)
im2col_rows_kernel(const uint4 *__restrict__ xp, int H, int W, int Ho, int Wo, int k, int s, int p, int d,
                   int cpp, Idx total, uint4 *__restrict__ rows) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t row_chunks = static_cast<int64_t>(k) * k * cpp;
    for (Idx t = static_cast<Idx>(blockIdx.x) * kPackThreads + threadIdx.x; t < total;
         t += static_cast<Idx>(gridDim.x) * kPackThreads) {
        const Idx m = t / static_cast<Idx>(cpp);
        const int c = static_cast<int>(t - m * static_cast<Idx>(cpp));
        const Idx r = m / static_cast<Idx>(Wo);
        const int wo = static_cast<int>(m - r * static_cast<Idx>(Wo));
        const Idx b = r / static_cast<Idx>(Ho);
        const int ho = static_cast<int>(r - b * static_cast<Idx>(Ho));
        const int h0 = ho * s - p, w0 = wo * s - p;
        const uint4 *src = xp + static_cast<int64_t>(b) * H * W * cpp + c;
        uint4 *dst = rows + static_cast<int64_t>(m) * row_chunks + c;
        for (int kh = 0; kh < k; ++kh) {
            const int hi = h0 + kh * d;
            const bool hin = hi >= 0 && hi < H;
#pragma unroll 4
            for (int kw = 0; kw < k; ++kw) {
                const int wi = w0 + kw * d;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (hin && wi >= 0 && wi < W) v = __ldg(src + (static_cast<int64_t>(hi) * W + wi) * cpp);
                dst[(kh * k + kw) * cpp] = v;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Fused shift + sign + pack + unfold for the tensor-core convolution: NCHW x
// straight to its im2col rows of packed codes. A unit is (image b, a band of
// hb output rows). TMA boxes bring the band's input rows into shared memory
// -- all channels; of each channel plane the band's pixels as one run from a
// 16-byte aligned pixel xa, in boxes of bw pixels x cbox channels; sign bits
// per (8-pixel group, channel) and the 8 x 8 bit transpose turn them into
// packed pixel codes in shared memory; then each output pixel's k*k taps
// leave as 16-byte stores of its im2col row, consecutive threads on
// consecutive chunks (zeros for a tap in the padding). The next unit's boxes
// are requested as soon as the band has been read.
// ---------------------------------------------------------------------------
constexpr int kUnfoldThreads = 256;

struct UnfoldArgs {
    int C, H, W, Ho, Wo, k, s, p, d;
    int hb, nbands;            // output rows per band, bands per image
    uint32_t units;            // B * nbands
    int bw, nxb;               // pixels per box (multiple of 32), boxes along the run
    int cbox, ncb;             // channels per box, boxes along the channels
    int span;                  // pixels staged per unit (nxb * bw)
    int cstride;               // bytes of a pixel group's row of sign bits
    int rbc, krow;             // bytes per packed pixel, per im2col row
    uint32_t box_bytes;        // bytes of one box
    uint32_t band_bytes;       // bytes of all boxes of a unit
    FastDiv div_nq;            // span / 32 pixel quads (32 pixels)
    FastDiv div_qpb;           // quads per box (bw / 32)
    FastDiv div_cbox;          // channels per box
    FastDiv div_g;             // 8-channel groups per packed pixel
    FastDiv div_rowc;          // 16-byte chunks per im2col row
    FastDiv div_cpp;           // 16-byte chunks per packed pixel
    FastDiv div_k, div_wo;
};

// Input rows [r_lo, r_hi] a band of output rows [ho0, ho1) reads, clipped to
// the image, and the aligned first pixel xa of its run.
__host__ __device__ __forceinline__ void unfold_band(const UnfoldArgs &u, int ho0, int ho1, int &r_lo, int &r_hi, int &xa) {
    r_lo = ho0 * u.s - u.p;
    r_hi = (ho1 - 1) * u.s - u.p + (u.k - 1) * u.d;
    if (r_lo < 0) r_lo = 0;
    if (r_lo > u.H - 1) r_lo = u.H - 1;
    if (r_hi > u.H - 1) r_hi = u.H - 1;
    xa = (r_lo * u.W) & ~7;
}

template <typename T, int CODE>
__global__ void __launch_bounds__(kUnfoldThreads)
pack_im2col_kernel(const __grid_constant__ CUtensorMap tmx, const UnfoldArgs u, const float *__restrict__ bias,
                   int bias_len, uint8_t *__restrict__ rows, unsigned int *err) {
    constexpr int OB = GroupOut<CODE>::kBytes;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *band = smem;
    uint8_t *sbits = smem + u.band_bytes;
    uint8_t *spix = sbits + (u.span / 8) * u.cstride;
    const uint32_t bar = smem_u32(spix + u.span * u.rbc);
    volatile uint32_t *flag = reinterpret_cast<volatile uint32_t *>(spix + u.span * u.rbc + 8);
    const int tid = threadIdx.x;
    const int npg = u.span / 8;
    const int G = static_cast<int>(u.div_g.d);
    const float bs = bias_len == 1 ? __ldg(bias) : 0.0f;

    if (tid == 0) {
        tc::mbar_init(bar, 1);
        *flag = 0u;
        tc::fence_mbar_init();
    }
    pdl_launch_dependents();
    __syncthreads();
    pdl_wait();                                          // x may come from, and rows go to, the previous kernel

    auto request = [&](uint32_t unit) {                  // thread 0: this unit's boxes
        const int b = static_cast<int>(unit / static_cast<uint32_t>(u.nbands));
        const int bnd = static_cast<int>(unit - static_cast<uint32_t>(b) * u.nbands);
        const int ho0 = bnd * u.hb, ho1 = ho0 + u.hb < u.Ho ? ho0 + u.hb : u.Ho;
        int r_lo, r_hi, xa;
        unfold_band(u, ho0, ho1, r_lo, r_hi, xa);
        tc::mbar_arrive_expect_tx(bar, u.band_bytes);
        for (int cb = 0; cb < u.ncb; ++cb)
            for (int xb = 0; xb < u.nxb; ++xb)
                tc::tma_load_2d(smem_u32(band) + static_cast<uint32_t>(cb * u.nxb + xb) * u.box_bytes, &tmx,
                                xa + xb * u.bw, b * u.C + cb * u.cbox, bar);
    };
    if (tid == 0 && blockIdx.x < u.units) request(blockIdx.x);

    uint32_t it = 0;
    for (uint32_t unit = blockIdx.x; unit < u.units; unit += gridDim.x, ++it) {
        const int b = static_cast<int>(unit / static_cast<uint32_t>(u.nbands));
        const int bnd = static_cast<int>(unit - static_cast<uint32_t>(b) * u.nbands);
        const int ho0 = bnd * u.hb, ho1 = ho0 + u.hb < u.Ho ? ho0 + u.hb : u.Ho;
        int r_lo, r_hi, xa;
        unfold_band(u, ho0, ho1, r_lo, r_hi, xa);
        if (tid == 0) (void)tc::wait_bounded(bar, it & 1u, flag, err);
        __syncthreads();
        if (*flag) break;
        (void)tc::mbar_try_wait(bar, it & 1u);           // completed phase: acquire for this thread

        // phase 1: sign bits, item (channel c, 32 pixels q4): four 8-pixel groups
        const int nq = u.span / 32;
        for (int i = tid; i < u.C * nq; i += kUnfoldThreads) {
            const int c = static_cast<int>(fdiv(static_cast<uint32_t>(i), u.div_nq));
            const int q4 = i - c * nq;
            const int cb = u.ncb == 1 ? 0 : static_cast<int>(fdiv(static_cast<uint32_t>(c), u.div_cbox));
            const int cl = c - cb * u.cbox;
            const int xb = u.nxb == 1 ? 0 : static_cast<int>(fdiv(static_cast<uint32_t>(q4), u.div_qpb));
            const int xl = 32 * q4 - xb * u.bw;
            const T *src = reinterpret_cast<const T *>(band + static_cast<uint32_t>(cb * u.nxb + xb) * u.box_bytes) +
                           cl * u.bw + xl;
            const float bc = bias_len > 1 ? __ldg(bias + c) : bs;
            const bool finite = isfinite(bc);
            uint8_t *dst = sbits + (4 * q4) * u.cstride + c;
#pragma unroll
            for (int g4 = 0; g4 < 4; ++g4) {
                Group<T> grp;
                grp.load_smem(src + 8 * g4);
                uint32_t P0, P1;
                if (finite) {
                    masks_ge<T>(grp, -bc, P0, P1);
                } else {
                    float f[8], bb[8];
                    grp.unpack(f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) bb[e] = bc;
                    masks_add(f, bb, P0, P1);
                }
                dst[g4 * u.cstride] = static_cast<uint8_t>(mask_byte(P0, P1));
            }
        }
        __syncthreads();
        // the band has been read: request the next unit's boxes
        if (tid == 0 && unit + gridDim.x < u.units) {
            tc::fence_proxy_async_smem();
            request(unit + gridDim.x);
        }

        // phase 2: packed pixel codes, item (pixel group pg, channel group cg)
        for (int i = tid; i < npg * G; i += kUnfoldThreads) {
            const int pg = static_cast<int>(fdiv(static_cast<uint32_t>(i), u.div_g));
            const int cg = i - pg * G;
            const int c0 = cg * 8;
            uint8_t *dst = spix + (8 * pg) * u.rbc + cg * OB;
            if (c0 >= u.C) {
#pragma unroll
                for (int j = 0; j < 8; ++j) store_group<CODE>(dst + j * u.rbc, 0u, 0u);
                continue;
            }
            const uint32_t cvalid = u.C - c0 >= 8 ? 0xFFu : (1u << (u.C - c0)) - 1u;
            const uint64_t v = transpose8x8(*reinterpret_cast<const uint64_t *>(sbits + pg * u.cstride + c0));
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t pos = static_cast<uint32_t>(v >> (8 * j)) & 0xFFu;
                store_group<CODE>(dst + j * u.rbc, ~pos & cvalid, cvalid);
            }
        }
        __syncthreads();

        // phase 3: im2col rows, item (output pixel, 16-byte chunk of its row)
        const int rowc = static_cast<int>(u.div_rowc.d), cpp = static_cast<int>(u.div_cpp.d);
        const int nopix = (ho1 - ho0) * u.Wo;
        for (int i = tid; i < nopix * rowc; i += kUnfoldThreads) {
            const int opix = static_cast<int>(fdiv(static_cast<uint32_t>(i), u.div_rowc));
            const int rc = i - opix * rowc;
            const int tap = static_cast<int>(fdiv(static_cast<uint32_t>(rc), u.div_cpp));
            const int chunk = rc - tap * cpp;
            const int kh = static_cast<int>(fdiv(static_cast<uint32_t>(tap), u.div_k));
            const int kw = tap - kh * u.k;
            const int oh = static_cast<int>(fdiv(static_cast<uint32_t>(opix), u.div_wo));
            const int wo = opix - oh * u.Wo;
            const int ho = ho0 + oh;
            const int hi = ho * u.s - u.p + kh * u.d, wi = wo * u.s - u.p + kw * u.d;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (hi >= 0 && hi < u.H && wi >= 0 && wi < u.W) {
                const int q = hi * u.W + wi - xa;
                v = *reinterpret_cast<const uint4 *>(spix + q * u.rbc + chunk * 16);
            }
            *reinterpret_cast<uint4 *>(rows + ((static_cast<int64_t>(b) * u.Ho + ho) * u.Wo + wo) * u.krow +
                                       rc * 16) = v;
        }
        __syncthreads();
    }
    if (tid == 0 && *flag) {
        // aborted: let a copy still in flight land before the CTA exits
        const unsigned long long t0 = globaltimer_ns();
        while (!tc::mbar_try_wait(bar, it & 1u) && globaltimer_ns() - t0 < kWaitNs) {}
    }
}

// The same result for any x layout (planes not 16-byte aligned): one thread
// per (output pixel m, tap, 8-channel group) reads its 8 channels straight
// from x and writes the group's code bytes; consecutive threads write
// consecutive groups of a row.
template <typename T, int CODE>
__global__ void __launch_bounds__(kPackThreads)
pack_im2col_direct_kernel(const T *__restrict__ x, int C, int H, int W, int Ho, int Wo, int k, int s, int p, int d,
                          FastDiv div_g, FastDiv div_kk, int krow, int64_t total, const float *__restrict__ bias,
                          int bias_len, uint8_t *__restrict__ rows) {
    constexpr int OB = GroupOut<CODE>::kBytes;
    pdl_launch_dependents();
    pdl_wait();
    const float bs = bias_len == 1 ? __ldg(bias) : 0.0f;
    const int G = static_cast<int>(div_g.d), kk = static_cast<int>(div_kk.d);
    const int64_t HW = static_cast<int64_t>(H) * W;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * kPackThreads + threadIdx.x; t < total;
         t += static_cast<int64_t>(gridDim.x) * kPackThreads) {
        const int64_t mt = t / G;                          // (m, tap)
        const int cg = static_cast<int>(t - mt * G);
        const int64_t m = mt / kk;
        const int tap = static_cast<int>(mt - m * kk);
        const int wo = static_cast<int>(m % Wo);
        const int64_t r = m / Wo;
        const int ho = static_cast<int>(r % Ho);
        const int64_t b = r / Ho;
        const int kh = tap / k, kw = tap - kh * k;
        const int hi = ho * s - p + kh * d, wi = wo * s - p + kw * d;
        const int c0 = cg * 8;
        uint32_t neg = 0, valid = 0;
        if (hi >= 0 && hi < H && wi >= 0 && wi < W) {
            const T *src = x + (b * C + c0) * HW + static_cast<int64_t>(hi) * W + wi;
            for (int e = 0; e < 8 && c0 + e < C; ++e) {
                const float bc = bias_len > 1 ? __ldg(bias + c0 + e) : bs;
                neg |= is_negative(Elem<T>::to_f32(src[e * HW]), bc) << e;
                valid |= 1u << e;
            }
        }
        store_group<CODE>(rows + m * krow + tap * (G * OB) + cg * OB, neg, valid);
    }
}

// For channel-packed pixels the warp-level kernels (contiguous loads) are the
// default where they apply (E2M1 from a 2-byte type: the conversion shared
// with the convolution's packing warps); BT_PACK_NHWC=smem selects the
// shared-memory transpose kernel and BT_PACK_NHWC=warp the byte-mask warp
// kernel for every code (all stay under test).
bool nhwc_warp_disabled() {
    const char *env = std::getenv("BT_PACK_NHWC");
    return env != nullptr && std::strcmp(env, "smem") == 0;
}
bool nhwc_e2m1_fast() {
    const char *env = std::getenv("BT_PACK_NHWC");
    return env == nullptr || (std::strcmp(env, "smem") != 0 && std::strcmp(env, "warp") != 0);
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
                   int64_t rb, cudaStream_t s, double *abs_sum = nullptr) {
    const int64_t G = padded_elems<CODE>(rb) / 8;
    const int64_t per_block = kRowThreads * kGroupsPerThread;
    dim3 grid(static_cast<unsigned>((G + per_block - 1) / per_block), static_cast<unsigned>(R < 65535 ? R : 65535));
    const bool vec = ((K * static_cast<int64_t>(sizeof(T))) % 16 == 0) && aligned(x, 16);
    const bool vec8 = ((K * static_cast<int64_t>(sizeof(T))) % 8 == 0) && aligned(x, 8);
    const int64_t total = R * G;
    const bool colbias = bias_len > 1;
    if (vec8 && total <= (int64_t(1) << 31) - (int64_t(1) << 21) && (!colbias || aligned(bias, 16))) {
        const int sms = device_sm_count();
        const int64_t per_block = kPackThreads * kFlatUnroll;
        const int64_t need = (total + per_block - 1) / per_block;
        const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 148) * (2048 / kPackThreads);
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute pdl = pdl_attribute();
        cfg.gridDim = dim3(static_cast<unsigned>(need < cap ? need : cap));
        cfg.blockDim = dim3(kPackThreads);
        cfg.stream = s;
        cfg.attrs = &pdl;
        cfg.numAttrs = 1;
        const FastDiv divG = make_fastdiv(static_cast<uint32_t>(G));
        const uint32_t Gf = static_cast<uint32_t>(K / 8);
        const uint32_t tot = static_cast<uint32_t>(total);
        const int k = static_cast<int>(K), bl = static_cast<int>(bias_len);
        if (abs_sum != nullptr) {
            // the same, adding the sum of |x| to *abs_sum
            if (vec)
                return colbias ? cudaLaunchKernelEx(&cfg, pack_rows_flat_kernel<T, CODE, true, 16, true>, x, tot, divG, Gf,
                                                    k, bias, bl, out, abs_sum)
                               : cudaLaunchKernelEx(&cfg, pack_rows_flat_kernel<T, CODE, false, 16, true>, x, tot, divG, Gf,
                                                    k, bias, bl, out, abs_sum);
            return colbias ? cudaLaunchKernelEx(&cfg, pack_rows_flat_kernel<T, CODE, true, 8, true>, x, tot, divG, Gf, k,
                                                bias, bl, out, abs_sum)
                           : cudaLaunchKernelEx(&cfg, pack_rows_flat_kernel<T, CODE, false, 8, true>, x, tot, divG, Gf,
                                                k, bias, bl, out, abs_sum);
        }
        if (vec)
            return colbias ? cudaLaunchKernelEx(&cfg, pack_rows_flat_kernel<T, CODE, true, 16>, x, tot, divG, Gf, k, bias, bl, out,
                                                static_cast<double *>(nullptr))
                           : cudaLaunchKernelEx(&cfg, pack_rows_flat_kernel<T, CODE, false, 16>, x, tot, divG, Gf, k, bias, bl, out,
                                                static_cast<double *>(nullptr));
        return colbias ? cudaLaunchKernelEx(&cfg, pack_rows_flat_kernel<T, CODE, true, 8>, x, tot, divG, Gf, k, bias, bl, out,
                                                static_cast<double *>(nullptr))
                       : cudaLaunchKernelEx(&cfg, pack_rows_flat_kernel<T, CODE, false, 8>, x, tot, divG, Gf, k, bias, bl, out,
                                                static_cast<double *>(nullptr));
    }
    if (abs_sum != nullptr) return cudaErrorNotSupported;
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
        const int sms = device_sm_count();
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
                   uint8_t *out, int64_t rb, cudaStream_t s, double *abs_sum = nullptr) {
    constexpr int E = Elem<T>::kPerVec;
    const bool vec = ((HW * static_cast<int64_t>(sizeof(T))) % 16 == 0) && aligned(x, 16);
    if (vec && HW < (int64_t(1) << 30) && C < (int64_t(1) << 30) && (abs_sum != nullptr || !nhwc_warp_disabled())) {
        // warp-level units of 32 channels x 256 pixels
        const int64_t npb = (HW + kWarpPackPixels - 1) / kWarpPackPixels, ncg = rb / Group32<CODE>::kBytes;
        const int64_t units = B * npb * ncg;
        if (units < (int64_t(1) << 31)) {
            const int sms = device_sm_count();
            const int64_t per_block = kPackThreads / 32;
            const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 148) * (2048 / kPackThreads);
            int64_t blocks = (units + per_block - 1) / per_block;
            if (blocks > cap) blocks = cap;
            if (blocks < 1) blocks = 1;
            // 2-byte inputs only: for f32 (two loads per 8 pixels) the byte-mask
            // kernel measured faster on GB300
            if (CODE == BT_CODE_E2M1 && sizeof(T) == 2 && abs_sum == nullptr && nhwc_e2m1_fast() &&
                (bias_len <= 1 || aligned(bias, 4))) {
                // pixel block fastest: unit u = (b * ncg + cg) * npb + blk; as many
                // blocks as are resident at once (the warps loop over the units), so
                // that no block waits for a second wave
                const FastDiv dncg = make_fastdiv(static_cast<uint32_t>(ncg)), dnpb = make_fastdiv(static_cast<uint32_t>(npb));
                auto kern = bias_len > 1 ? pack_nhwc_e2m1_kernel<T, true> : pack_nhwc_e2m1_kernel<T, false>;
                static int per_sm[2] = {0, 0};
                const int slot = bias_len > 1 ? 1 : 0;
                if (per_sm[slot] == 0) {
                    int n = 0;
                    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kPackThreads, 0) != cudaSuccess || n < 1) n = 1;
                    per_sm[slot] = n;
                }
                int64_t eb = static_cast<int64_t>(sms > 0 ? sms : 148) * per_sm[slot];
                const int64_t need = (units + per_block - 1) / per_block;
                if (eb > need) eb = need;
                if (eb < 1) eb = 1;
                return launch_pdl(kern, dim3(static_cast<unsigned>(eb)), dim3(kPackThreads), s, x, static_cast<int>(C),
                                  static_cast<int>(HW), static_cast<uint32_t>(units), dncg, dnpb, bias,
                                  static_cast<int>(bias_len), out, static_cast<int>(rb));
            }
            if (abs_sum != nullptr)
                return launch_pdl(pack_nhwc_warp_kernel<T, CODE, true>, dim3(static_cast<unsigned>(blocks)),
                                  dim3(kPackThreads), s, x, static_cast<int>(C), static_cast<int>(HW),
                                  static_cast<uint32_t>(units), make_fastdiv(static_cast<uint32_t>(npb)),
                                  make_fastdiv(static_cast<uint32_t>(ncg)), bias, static_cast<int>(bias_len), out,
                                  static_cast<int>(rb), abs_sum);
            return launch_pdl(pack_nhwc_warp_kernel<T, CODE>, dim3(static_cast<unsigned>(blocks)), dim3(kPackThreads),
                              s, x, static_cast<int>(C), static_cast<int>(HW), static_cast<uint32_t>(units),
                              make_fastdiv(static_cast<uint32_t>(npb)), make_fastdiv(static_cast<uint32_t>(ncg)), bias,
                              static_cast<int>(bias_len), out, static_cast<int>(rb), static_cast<double *>(nullptr));
        }
    }
    if (abs_sum != nullptr) return cudaErrorNotSupported;
    const int smem = kNhwcGroups * nhwc_cstride(static_cast<int>(C));
    const int64_t upi = (HW + kNhwcPixels - 1) / kNhwcPixels;
    const int64_t G = padded_elems<CODE>(rb) / 8;
    if (smem <= kNhwcMaxSmem && B * upi < (int64_t(1) << 31) && G * kNhwcGroups < (int64_t(1) << 31)) {
        const int sms = device_sm_count();
        const int64_t units = B * upi;
        const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 148) * (2048 / kPackThreads);
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute pdl = pdl_attribute();
        cfg.gridDim = dim3(static_cast<unsigned>(units < cap ? units : cap));
        cfg.blockDim = dim3(kPackThreads);
        cfg.dynamicSmemBytes = static_cast<size_t>(smem);
        cfg.stream = s;
        cfg.attrs = &pdl;
        cfg.numAttrs = 1;
        const FastDiv divG = make_fastdiv(static_cast<uint32_t>(G));
        if (vec)
            return cudaLaunchKernelEx(&cfg, pack_nhwc_tr_kernel<T, CODE, true>, x, static_cast<int>(C),
                                      static_cast<int>(HW), static_cast<int>(upi), static_cast<uint32_t>(units), bias,
                                      static_cast<int>(bias_len), out, static_cast<int>(rb), divG);
        return cudaLaunchKernelEx(&cfg, pack_nhwc_tr_kernel<T, CODE, false>, x, static_cast<int>(C),
                                  static_cast<int>(HW), static_cast<int>(upi), static_cast<uint32_t>(units), bias,
                                  static_cast<int>(bias_len), out, static_cast<int>(rb), divG);
    }
    const int64_t threads = B * (padded_elems<CODE>(rb) / 8) * ((HW + E - 1) / E);
    const int grid = grid_for(threads);
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
                      void *out, cudaStream_t s, double *abs_sum = nullptr) {
    uint8_t *o = static_cast<uint8_t *>(out);
    const int64_t rb = row_bytes(K, code);
    switch (code) {
        case BT_CODE_BITS: return rows_t<T, BT_CODE_BITS>(x, R, K, bias, bias_len, o, rb, s, abs_sum);
        case BT_CODE_E4M3: return rows_t<T, BT_CODE_E4M3>(x, R, K, bias, bias_len, o, rb, s, abs_sum);
        default: return rows_t<T, BT_CODE_E2M1>(x, R, K, bias, bias_len, o, rb, s, abs_sum);
    }
}

template <typename T>
cudaError_t nhwc_code(const T *x, int64_t B, int64_t C, int64_t HW, const float *bias, int64_t bias_len,
                      bt_code code, void *out, cudaStream_t s, double *abs_sum = nullptr) {
    uint8_t *o = static_cast<uint8_t *>(out);
    const int64_t rb = row_bytes(C, code);
    switch (code) {
        case BT_CODE_BITS: return nhwc_t<T, BT_CODE_BITS>(x, B, C, HW, bias, bias_len, o, rb, s, abs_sum);
        case BT_CODE_E4M3: return nhwc_t<T, BT_CODE_E4M3>(x, B, C, HW, bias, bias_len, o, rb, s, abs_sum);
        default: return nhwc_t<T, BT_CODE_E2M1>(x, B, C, HW, bias, bias_len, o, rb, s, abs_sum);
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

cudaError_t launch_pack_rows_sum(const void *x, bt_dtype xt, int64_t R, int64_t K, const float *bias,
                                 int64_t bias_len, bt_code code, void *out, double *abs_sum, cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    switch (xt) {
        case BT_F32: return rows_code(static_cast<const float *>(x), R, K, bias, bias_len, code, out, s, abs_sum);
        case BT_BF16:
            return rows_code(static_cast<const __nv_bfloat16 *>(x), R, K, bias, bias_len, code, out, s, abs_sum);
        default: return rows_code(static_cast<const __half *>(x), R, K, bias, bias_len, code, out, s, abs_sum);
    }
}

namespace {

constexpr int kUnfoldMaxSmem = 113 * 1024;              // two units' worth of CTAs per SM

template <typename T> CUtensorMapDataType map_type();
template <> CUtensorMapDataType map_type<float>() { return CU_TENSOR_MAP_DATA_TYPE_FLOAT32; }
template <> CUtensorMapDataType map_type<__nv_bfloat16>() { return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16; }
template <> CUtensorMapDataType map_type<__half>() { return CU_TENSOR_MAP_DATA_TYPE_FLOAT16; }

int unfold_smem(const UnfoldArgs &u) {
    return static_cast<int>(u.band_bytes) + (u.span / 8) * u.cstride + u.span * u.rbc + 16;
}

// Plan the staged unfold of a problem: the band height and boxes (see
// UnfoldArgs). False when x's planes are not 16-byte aligned or no band fits.
// `efficient` tells whether the plan runs at least three CTAs per SM and
// stages at most 1.3x the input (measured on GB300: then one pass beats
// packing pixels and unfolding them in a second kernel).
bool plan_unfold(const ConvGeom &g, int elem, bt_code code, UnfoldArgs &out, bool &efficient) {
    const int64_t HW = g.H * g.W;
    if ((HW * elem) % 16 != 0 || g.C > 16384 || g.B * g.C > (int64_t(1) << 31)) return false;
    UnfoldArgs u{};
    u.C = static_cast<int>(g.C); u.H = static_cast<int>(g.H); u.W = static_cast<int>(g.W);
    u.Ho = static_cast<int>(g.Ho); u.Wo = static_cast<int>(g.Wo);
    u.k = g.k; u.s = g.s; u.p = g.p; u.d = g.d;
    u.rbc = static_cast<int>(row_bytes(g.C, code));
    u.krow = g.k * g.k * u.rbc;
    u.ncb = static_cast<int>((g.C + 255) / 256);
    u.cbox = static_cast<int>((g.C + u.ncb - 1) / u.ncb);
    u.cstride = static_cast<int>((g.C + 7) / 8 * 8 + 8);
    const int sms = device_sm_count();
    // the tallest band that leaves two units per SM within a staging budget,
    // trying budgets of four, three and two CTAs per SM in turn (else the
    // shortest band that fits the largest budget)
    bool found = false;
    UnfoldArgs best{};
    int64_t best_rows_in = 0;
    const int budgets[3] = {54 * 1024, 74 * 1024, kUnfoldMaxSmem};
    for (int bi = 0; bi < 3 && !found; ++bi) {
        for (int hb = u.Ho; hb >= 1; --hb) {
            int64_t rows_in = static_cast<int64_t>(hb - 1) * g.s + static_cast<int64_t>(g.k - 1) * g.d + 1;
            if (rows_in > g.H) rows_in = g.H;
            const int64_t need = rows_in * g.W + 7;
            const int64_t nxb = (need + 255) / 256;
            const int64_t bw = ((need + nxb - 1) / nxb + 31) / 32 * 32;
            if (bw > 256 || nxb > 16) continue;
            UnfoldArgs c = u;
            c.hb = hb;
            c.nbands = (u.Ho + hb - 1) / hb;
            c.nxb = static_cast<int>(nxb);
            c.bw = static_cast<int>(bw);
            c.span = static_cast<int>(nxb * bw);
            c.box_bytes = static_cast<uint32_t>(c.cbox * c.bw * elem);
            c.band_bytes = c.box_bytes * static_cast<uint32_t>(c.ncb * c.nxb);
            if (unfold_smem(c) > budgets[bi]) continue;
            const int64_t units = g.B * c.nbands;
            if (units >= 2LL * sms) { best = c; best_rows_in = rows_in; found = true; break; }
            if (bi == 2) { best = c; best_rows_in = rows_in; found = true; }   // keep shrinking: more units
        }
    }
    if (!found || g.B * best.nbands > (int64_t(1) << 31) - 1) return false;
    const int per_sm = (227 * 1024) / (unfold_smem(best) + 1024);
    const double overread = static_cast<double>(best.nbands) * static_cast<double>(best_rows_in) / static_cast<double>(g.H);
    efficient = per_sm >= 3 && overread <= 1.3;
    out = best;
    return true;
}

template <typename T, int CODE>
cudaError_t im2col_t(const T *x, const ConvGeom &g, const float *bias, int64_t bias_len, uint8_t *rows,
                     bool efficient_only, cudaStream_t s) {
    constexpr int elem = static_cast<int>(sizeof(T));
    const int64_t HW = g.H * g.W;
    auto enc = tensor_map_encoder();
    UnfoldArgs u{};
    bool efficient = false;
    if (enc == nullptr || !aligned(x, 16) || !plan_unfold(g, elem, static_cast<bt_code>(CODE), u, efficient) ||
        (efficient_only && !efficient))
        return cudaErrorNotSupported;
    const int sms = device_sm_count();
    u.units = static_cast<uint32_t>(g.B * u.nbands);
    u.div_nq = make_fastdiv(static_cast<uint32_t>(u.span / 32));
    u.div_qpb = make_fastdiv(static_cast<uint32_t>(u.bw / 32));
    u.div_cbox = make_fastdiv(static_cast<uint32_t>(u.cbox));
    u.div_g = make_fastdiv(static_cast<uint32_t>(u.rbc / GroupOut<CODE>::kBytes));
    u.div_rowc = make_fastdiv(static_cast<uint32_t>(u.krow / 16));
    u.div_cpp = make_fastdiv(static_cast<uint32_t>(u.rbc / 16));
    u.div_k = make_fastdiv(static_cast<uint32_t>(g.k));
    u.div_wo = make_fastdiv(static_cast<uint32_t>(g.Wo));

    // x as a 2-D tensor [B*C planes, H*W pixels]; boxes of bw pixels x cbox channels, zero fill outside
    CUtensorMap m;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(HW), static_cast<cuuint64_t>(g.B * g.C)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(HW * elem)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(u.bw), static_cast<cuuint32_t>(u.cbox)};
    cuuint32_t estr[2] = {1, 1};
    if (enc(&m, map_type<T>(), 2, const_cast<T *>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
        return cudaErrorNotSupported;

    unsigned int *err = device_error_word();
    if (err == nullptr) return cudaErrorUnknown;
    auto kern = pack_im2col_kernel<T, CODE>;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [&] { attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kUnfoldMaxSmem); });
    if (attr != cudaSuccess) return attr;
    const int smem = unfold_smem(u);
    int per_sm = (227 * 1024) / (smem + 1024);
    if (per_sm < 1) per_sm = 1;
    const int64_t cap = static_cast<int64_t>(sms) * per_sm;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute pdl = pdl_attribute();
    cfg.gridDim = dim3(static_cast<unsigned>(u.units < cap ? u.units : cap));
    cfg.blockDim = dim3(kUnfoldThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cfg.attrs = &pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, m, u, bias, static_cast<int>(bias_len), rows, err);
}

template <typename T, int CODE>
cudaError_t im2col_direct_t(const T *x, const ConvGeom &g, const float *bias, int64_t bias_len, uint8_t *rows,
                            cudaStream_t s) {
    const int64_t rbc = row_bytes(g.C, static_cast<bt_code>(CODE));
    const int G = static_cast<int>(rbc / GroupOut<CODE>::kBytes), kk = g.k * g.k;
    const int64_t total = g.B * g.Ho * g.Wo * kk * G;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * (2048 / kPackThreads);
    const int64_t blocks = (total + kPackThreads - 1) / kPackThreads;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute pdl = pdl_attribute();
    cfg.gridDim = dim3(static_cast<unsigned>(blocks < cap ? blocks : cap));
    cfg.blockDim = dim3(kPackThreads);
    cfg.stream = s;
    cfg.attrs = &pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, pack_im2col_direct_kernel<T, CODE>, x, static_cast<int>(g.C), static_cast<int>(g.H),
                              static_cast<int>(g.W), static_cast<int>(g.Ho), static_cast<int>(g.Wo), g.k, g.s, g.p, g.d,
                              make_fastdiv(static_cast<uint32_t>(G)), make_fastdiv(static_cast<uint32_t>(kk)),
                              static_cast<int>(kk * rbc), total, bias, static_cast<int>(bias_len), rows);
}

template <typename T>
cudaError_t im2col_code(const T *x, const ConvGeom &g, const float *bias, int64_t bias_len, bt_code code,
                        uint8_t *rows, bool direct_ok, cudaStream_t s) {
    // direct_ok: a public unfold call (any plan, else the direct kernel);
    // otherwise the convolution asks for the one-pass unfold only where it pays
    cudaError_t e = cudaErrorNotSupported;
    if (code == BT_CODE_E4M3) e = im2col_t<T, BT_CODE_E4M3>(x, g, bias, bias_len, rows, !direct_ok, s);
    else if (code == BT_CODE_E2M1) e = im2col_t<T, BT_CODE_E2M1>(x, g, bias, bias_len, rows, !direct_ok, s);
    if (e != cudaErrorNotSupported || !direct_ok) return e;
    if (code == BT_CODE_E4M3) return im2col_direct_t<T, BT_CODE_E4M3>(x, g, bias, bias_len, rows, s);
    if (code == BT_CODE_E2M1) return im2col_direct_t<T, BT_CODE_E2M1>(x, g, bias, bias_len, rows, s);
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_pack_im2col(const void *x, bt_dtype xt, const ConvGeom &g, const float *bias, int64_t bias_len,
                               bt_code code, uint8_t *rows, bool direct_ok, cudaStream_t s) {
    if (g.B == 0 || g.Ho * g.Wo == 0) return cudaSuccess;
    switch (xt) {
        case BT_F32: return im2col_code(static_cast<const float *>(x), g, bias, bias_len, code, rows, direct_ok, s);
        case BT_BF16:
            return im2col_code(static_cast<const __nv_bfloat16 *>(x), g, bias, bias_len, code, rows, direct_ok, s);
        case BT_F16: return im2col_code(static_cast<const __half *>(x), g, bias, bias_len, code, rows, direct_ok, s);
        default: return cudaErrorNotSupported;
    }
}

bool unfold_single_pass(const ConvGeom &g, bt_dtype xt, bt_code code) {
    if ((code != BT_CODE_E4M3 && code != BT_CODE_E2M1) || tensor_map_encoder() == nullptr) return false;
    UnfoldArgs u{};
    bool efficient = false;
    return plan_unfold(g, dtype_bytes(xt), code, u, efficient) && efficient;
}

cudaError_t launch_im2col_rows(const uint8_t *xp, const ConvGeom &g, int64_t rbc, uint8_t *rows, cudaStream_t s) {
    const int64_t M = g.B * g.Ho * g.Wo;
    if (M == 0) return cudaSuccess;
    const int cpp = static_cast<int>(rbc / 16);
    const int64_t total = M * cpp;
    const int sms = device_sm_count();
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 148) * 8;
    const int64_t blocks = (total + kPackThreads - 1) / kPackThreads;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute pdl = pdl_attribute();
    cfg.gridDim = dim3(static_cast<unsigned>(blocks < cap ? blocks : cap));
    cfg.blockDim = dim3(kPackThreads);
    cfg.stream = s;
    cfg.attrs = &pdl;
    cfg.numAttrs = 1;
    const uint4 *src = reinterpret_cast<const uint4 *>(xp);
    uint4 *dst = reinterpret_cast<uint4 *>(rows);
    const int H = static_cast<int>(g.H), W = static_cast<int>(g.W), Ho = static_cast<int>(g.Ho),
              Wo = static_cast<int>(g.Wo);
    if (total < (int64_t(1) << 32) - kPackThreads * cap)
        return cudaLaunchKernelEx(&cfg, im2col_rows_kernel<uint32_t>, src, H, W, Ho, Wo, g.k, g.s, g.p, g.d, cpp,
                                  static_cast<uint32_t>(total), dst);
    return cudaLaunchKernelEx(&cfg, im2col_rows_kernel<uint64_t>, src, H, W, Ho, Wo, g.k, g.s, g.p, g.d, cpp,
                              static_cast<uint64_t>(total), dst);
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

cudaError_t launch_pack_nhwc_sum(const void *x, bt_dtype xt, int64_t B, int64_t C, int64_t HW, const float *bias,
                                 int64_t bias_len, bt_code code, void *out, double *abs_sum, cudaStream_t s) {
    if (B == 0) return cudaSuccess;
    switch (xt) {
        case BT_F32: return nhwc_code(static_cast<const float *>(x), B, C, HW, bias, bias_len, code, out, s, abs_sum);
        case BT_BF16:
            return nhwc_code(static_cast<const __nv_bfloat16 *>(x), B, C, HW, bias, bias_len, code, out, s, abs_sum);
        default: return nhwc_code(static_cast<const __half *>(x), B, C, HW, bias, bias_len, code, out, s, abs_sum);
    }
}

}  // namespace bt
