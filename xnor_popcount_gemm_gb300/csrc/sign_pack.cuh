// Sign-mask and bit-transpose helpers shared by the standalone pack kernels
// and the convolution that packs its own input: the activation shift + sign of
// bitorch-engine BinaryConv2dCutlass.set_activation / the native forward,
// evaluated exactly, eight values at a time.
#pragma once

#include <cstdint>

#include "bt_device.cuh"

namespace bt {

// One group of 8 elements as 2 * sizeof(T) 32-bit words (value e of a 2-byte
// type in half e % 2 of word e / 2), loaded with VB-byte vectors (16 or 8;
// the group's address must be VB-aligned).
template <typename T> struct Group {
    static constexpr int kWords = 2 * static_cast<int>(sizeof(T));
    uint32_t w[kWords];
    template <int VB = 16>
    __device__ __forceinline__ void load(const T *p) {
        if constexpr (VB == 16) {
#pragma unroll
            for (int i = 0; i < kWords / 4; ++i) {
                const uint4 q = ld_stream_v4(p + i * (16 / sizeof(T)));
                w[4 * i] = q.x; w[4 * i + 1] = q.y; w[4 * i + 2] = q.z; w[4 * i + 3] = q.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < kWords / 2; ++i) {
                const uint2 q = __ldcs(reinterpret_cast<const uint2 *>(p + i * (8 / sizeof(T))));
                w[2 * i] = q.x; w[2 * i + 1] = q.y;
            }
        }
    }
    __device__ __forceinline__ void load_smem(const T *p) {     // 16-byte aligned shared memory
#pragma unroll
        for (int i = 0; i < kWords / 4; ++i) {
            const uint4 q = *reinterpret_cast<const uint4 *>(p + i * (16 / sizeof(T)));
            w[4 * i] = q.x; w[4 * i + 1] = q.y; w[4 * i + 2] = q.z; w[4 * i + 3] = q.w;
        }
    }
    __device__ __forceinline__ void unpack(float (&f)[8]) const {
#pragma unroll
        for (int i = 0; i < kWords / 4; ++i)
            Elem<T>::unpack(make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]), f + i * Elem<T>::kPerVec);
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

// ---------------------------------------------------------------------------
// Sign masks. For a finite shift b, x + b >= 0 (the fp32 sum, exact in sign)
// holds exactly when x >= -b, and for x of a 2-byte type exactly when x >= t
// with t = -b rounded up to that type (the smallest value of the type that is
// >= -b; +inf past its range). So 2-byte inputs are compared two at a time
// against t, without widening. A non-finite b takes the fp32 sum itself.
// The masks come out as two words P0 (values 0..3) and P1 (values 4..7), byte
// e 0xFF where value e binarizes to +1, else 0.
// ---------------------------------------------------------------------------
template <typename T> struct Thresh;
template <> struct Thresh<__nv_bfloat16> {
    using type = __nv_bfloat162;
    __device__ __forceinline__ static type of(float neg_b) {
        const __nv_bfloat16 t = __float2bfloat16_ru(neg_b);
        return __halves2bfloat162(t, t);
    }
    __device__ __forceinline__ static uint32_t ge(uint32_t w, type t) {
        return __hge2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&w), t);
    }
};
template <> struct Thresh<__half> {
    using type = __half2;
    __device__ __forceinline__ static type of(float neg_b) {
        const __half t = __float2half_ru(neg_b);
        return __halves2half2(t, t);
    }
    __device__ __forceinline__ static uint32_t ge(uint32_t w, type t) {
        return __hge2_mask(*reinterpret_cast<const __half2 *>(&w), t);
    }
};

// Masks of one group from its 16-byte (2-byte types) or 2 x 16-byte (fp32)
// loads against a threshold (finite shift).
template <typename T>
__device__ __forceinline__ void masks_ge(const Group<T> &g, float neg_b, uint32_t &P0, uint32_t &P1) {
    if constexpr (sizeof(T) == 2) {
        const typename Thresh<T>::type t = Thresh<T>::of(neg_b);
        const uint32_t m0 = Thresh<T>::ge(g.w[0], t), m1 = Thresh<T>::ge(g.w[1], t);
        const uint32_t m2 = Thresh<T>::ge(g.w[2], t), m3 = Thresh<T>::ge(g.w[3], t);
        P0 = __byte_perm(m0, m1, 0x6420);
        P1 = __byte_perm(m2, m3, 0x6420);
    } else {
        uint32_t s[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) s[e] = __uint_as_float(g.w[e]) >= neg_b ? 0xFFFFFFFFu : 0u;
        P0 = __byte_perm(__byte_perm(s[0], s[1], 0x0040), __byte_perm(s[2], s[3], 0x0040), 0x5410);
        P1 = __byte_perm(__byte_perm(s[4], s[5], 0x0040), __byte_perm(s[6], s[7], 0x0040), 0x5410);
    }
}

// The same from the fp32 sums x + b (any shift, one per value).
__device__ __forceinline__ void masks_add(const float (&f)[8], const float (&b)[8], uint32_t &P0, uint32_t &P1) {
    uint32_t s[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) s[e] = is_negative(f[e], b[e]) ? 0u : 0xFFFFFFFFu;
    P0 = __byte_perm(__byte_perm(s[0], s[1], 0x0040), __byte_perm(s[2], s[3], 0x0040), 0x5410);
    P1 = __byte_perm(__byte_perm(s[4], s[5], 0x0040), __byte_perm(s[6], s[7], 0x0040), 0x5410);
}

// One byte, bit e set where value e binarizes to +1: one bit gathered from
// each mask byte with a multiply (the four partial products land on distinct
// bits, so nothing carries).
__device__ __forceinline__ uint32_t mask_byte(uint32_t P0, uint32_t P1) {
    const uint32_t lo = ((P0 & 0x08040201u) * 0x01010101u) >> 24;
    const uint32_t hi = ((P1 & 0x08040201u) * 0x01010101u) >> 24;
    return lo | (hi << 4);
}

// One exchange round: swaps, between lanes l and l ^ L, the bits whose lane bit
// (weight L) differs from their register bit (weight R): afterwards bit (lane,
// reg) holds what bit (lane with its L-bit set to reg's R-bit, reg with its
// R-bit set to lane's L-bit) held. M: the register bits whose R-bit is 0.
template <int L, int R, uint32_t M>
__device__ __forceinline__ uint32_t exchange_bits(uint32_t w, int lane) {
    const uint32_t t = __shfl_xor_sync(0xFFFFFFFFu, w, L);
    return (lane & L) ? ((w & ~M) | ((t >> R) & M)) : ((w & M) | ((t & M) << R));
}

}  // namespace bt
