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

// A 16-byte load through the non-coherent path, issued where it stands in
// the program (volatile: the pack loop relies on its loads going out ahead of
// the conversion of earlier units).
__device__ __forceinline__ uint4 ld_nc_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// One bit-matrix exchange round across a warp, rotate form: swaps between
// lanes l and l ^ L the bits whose lane bit L differs from their register bit
// of weight R (R = L here). `keep` (the positions this lane keeps: R-bit equal
// to its L-bit) and `rot` (R, or 32 - R where the L-bit is clear) are fixed per
// lane. A shuffle, a funnel shift and one three-input logic op.
__device__ __forceinline__ uint32_t exchange_rot(uint32_t w, int L, uint32_t keep, uint32_t rot) {
    const uint32_t t = __shfl_xor_sync(0xFFFFFFFFu, w, L);
    const uint32_t r = __funnelshift_r(t, t, rot);
    return (w & keep) | (r & ~keep);
}

// A load of 16 bytes that only goes out where `ok` holds (zeros otherwise):
// predicated in place, no branch.
__device__ __forceinline__ uint4 ld_nc_v4_if(const void *p, bool ok) {
    uint4 v;
    asm volatile(
        "{\n .reg .pred q;\n setp.ne.b32 q, %5, 0;\n"
        " mov.b32 %0, 0;\n mov.b32 %1, 0;\n mov.b32 %2, 0;\n mov.b32 %3, 0;\n"
        " @q ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];\n}"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p), "r"(static_cast<int>(ok)));
    return v;
}

// The sign test of the shift as one comparison x >= t (the activation shift
// of BinaryConv2dCutlass.set_activation: +1 where x + b >= 0, the fp32 sum).
// A finite b: t = -b, rounded up to a 2-byte input type (x + b >= 0 exactly
// when x >= -b; for a 2-byte x exactly when x >= that rounding). b = +inf:
// x + b >= 0 for every x but -inf and NaN, i.e. x >= the lowest finite value.
// b = -inf or NaN: never, i.e. x >= NaN. Returned as the comparison operand's
// bits: the value in both halves for a 2-byte type, the float for f32.
template <typename XT> __device__ __forceinline__ uint32_t shift_threshold(float b);
template <> __device__ __forceinline__ uint32_t shift_threshold<float>(float b) {
    if (isfinite(b)) return __float_as_uint(-b);
    return b > 0.0f ? 0xFF7FFFFFu : 0x7FC00000u;
}
template <> __device__ __forceinline__ uint32_t shift_threshold<__nv_bfloat16>(float b) {
    if (isfinite(b)) {
        const __nv_bfloat16 t = __float2bfloat16_ru(-b);
        const uint32_t h = *reinterpret_cast<const uint16_t *>(&t);
        return h | (h << 16);
    }
    return b > 0.0f ? 0xFF7FFF7Fu : 0x7FC07FC0u;
}
template <> __device__ __forceinline__ uint32_t shift_threshold<__half>(float b) {
    if (isfinite(b)) {
        const __half t = __float2half_ru(-b);
        const uint32_t h = *reinterpret_cast<const uint16_t *>(&t);
        return h | (h << 16);
    }
    return b > 0.0f ? 0xFBFFFBFFu : 0x7E007E00u;
}

// Sign bits of one load group (8 consecutive pixels of one channel, k = the
// channel's bits 4..3) at register bit 16*p0 + 8*p2 + 4*p1 + k, p the pixel
// within the group: with a 2-byte type each pair of values is one comparison
// whose two 16-bit halves land on the pair's two bits.
template <typename XT>
__device__ __forceinline__ uint32_t sign_bits(const uint4 &lo, const uint4 &hi, uint32_t t, int k) {
    uint32_t w = 0;
    if constexpr (sizeof(XT) == 2) {
        using T2 = typename Thresh<XT>::type;
        const T2 tt = *reinterpret_cast<const T2 *>(&t);
        w |= Thresh<XT>::ge(lo.x, tt) & (0x00010001u << k);
        w |= Thresh<XT>::ge(lo.y, tt) & (0x00010001u << (4 + k));
        w |= Thresh<XT>::ge(lo.z, tt) & (0x00010001u << (8 + k));
        w |= Thresh<XT>::ge(lo.w, tt) & (0x00010001u << (12 + k));
    } else {
        const float tf = __uint_as_float(t);
        const uint32_t v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
        for (int e = 0; e < 8; ++e)
            w |= (__uint_as_float(v[e]) >= tf ? 1u : 0u) << (16 * (e & 1) + 4 * (e >> 1) + k);
    }
    return w;
}

}  // namespace bt
