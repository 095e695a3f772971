// Device-side helpers shared by the kernels of libbt.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "bt.h"

namespace bt {

// Error-word bits. A kernel ORs one in and returns; it never traps.
constexpr unsigned int kErrTimeout = 1u;

// ---------------------------------------------------------------------------
// Binarization: +1 where x + bias >= 0. The fp32 sum is exact in sign (without
// flushing subnormals, the exact sum of two floats never rounds to zero), so
// this is the sign of the exact sum; -0.0 gives +1, NaN gives -1.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t sign_bit(float v, float b) {
    return __fadd_rn(v, b) >= 0.0f ? 1u : 0u;
}
// The complement: 1 where the value binarizes to -1.
__device__ __forceinline__ uint32_t is_negative(float v, float b) {
    return __fadd_rn(v, b) >= 0.0f ? 0u : 1u;
}

// Codes of +1 / -1.
constexpr uint32_t kE4M3Plus = 0x38u, kE4M3Minus = 0xB8u;
constexpr uint32_t kE2M1Plus = 0x2u, kE2M1Minus = 0xAu;

__device__ __forceinline__ uint32_t e4m3_code(uint32_t bit) { return bit ? kE4M3Plus : kE4M3Minus; }
__device__ __forceinline__ uint32_t e2m1_code(uint32_t bit) { return bit ? kE2M1Plus : kE2M1Minus; }

// Element loads converted exactly to fp32.
template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kPerVec = 4;
    __device__ __forceinline__ static float to_f32(float v) { return v; }
    __device__ __forceinline__ static void unpack(const uint4 &q, float *f) {
        f[0] = __uint_as_float(q.x); f[1] = __uint_as_float(q.y);
        f[2] = __uint_as_float(q.z); f[3] = __uint_as_float(q.w);
    }
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int kPerVec = 8;
    __device__ __forceinline__ static float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ __forceinline__ static void unpack(const uint4 &q, float *f) {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
};
template <> struct Elem<__half> {
    static constexpr int kPerVec = 8;
    __device__ __forceinline__ static float to_f32(__half v) { return __half2float(v); }
    __device__ __forceinline__ static void unpack(const uint4 &q, float *f) {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
            float2 t = __half22float2(h);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
};

// Streaming 16-byte load (read once, do not keep in L1).
__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}

// ---------------------------------------------------------------------------
// Epilogue: y = fp32(dot * alpha) (one rounding), cast to the output type.
// ---------------------------------------------------------------------------
template <int OUT> struct OutT;
template <> struct OutT<BT_F32> {
    using type = float;
    __device__ __forceinline__ static float cvt(int dot, float alpha) {
        return __fmul_rn(static_cast<float>(dot), alpha);
    }
};
template <> struct OutT<BT_BF16> {
    using type = __nv_bfloat16;
    __device__ __forceinline__ static __nv_bfloat16 cvt(int dot, float alpha) {
        return __float2bfloat16_rn(__fmul_rn(static_cast<float>(dot), alpha));
    }
};
template <> struct OutT<BT_F16> {
    using type = __half;
    __device__ __forceinline__ static __half cvt(int dot, float alpha) {
        return __float2half_rn(__fmul_rn(static_cast<float>(dot), alpha));
    }
};
template <> struct OutT<BT_I32> {
    using type = int;
    __device__ __forceinline__ static int cvt(int dot, float) { return dot; }
};

// The same from a tensor-core accumulator: the fp32 accumulator already holds
// the exact integer dot (|dot| < 2^24), so fp32(dot * alpha) is one multiply
// of it -- no integer round trip.
template <int OUT> struct FromAcc;
template <> struct FromAcc<BT_F32> {
    __device__ __forceinline__ static uint32_t bits(float acc, float alpha) {
        return __float_as_uint(__fmul_rn(acc, alpha));
    }
};
template <> struct FromAcc<BT_I32> {
    __device__ __forceinline__ static uint32_t bits(float acc, float) {
        return static_cast<uint32_t>(__float2int_rn(acc));
    }
};
// Two 16-bit outputs packed in one word (first in the low half).
template <int OUT> __device__ __forceinline__ uint32_t pack2_from_acc(float a0, float a1, float alpha);
template <> __device__ __forceinline__ uint32_t pack2_from_acc<BT_BF16>(float a0, float a1, float alpha) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(__fmul_rn(a0, alpha), __fmul_rn(a1, alpha));
    return *reinterpret_cast<const uint32_t *>(&v);
}
template <> __device__ __forceinline__ uint32_t pack2_from_acc<BT_F16>(float a0, float a1, float alpha) {
    const __half2 v = __floats2half2_rn(__fmul_rn(a0, alpha), __fmul_rn(a1, alpha));
    return *reinterpret_cast<const uint32_t *>(&v);
}

// Division by a divisor fixed per launch, for n < 2^31: q = (hi32(m*n) + n) >> l
// with l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1 (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994).
struct FastDiv {
    uint32_t d, m, l;
};
inline FastDiv make_fastdiv(uint32_t d) {
    uint32_t l = 0;
    while ((uint64_t(1) << l) < d) ++l;
    const uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1;
    return FastDiv{d, static_cast<uint32_t>(m), l};
}
__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f) { return (__umulhi(f.m, n) + n) >> f.l; }

// ---------------------------------------------------------------------------
// Bounded waiting. Every spin in these kernels gives up after kWaitNs of
// %globaltimer time, records kErrTimeout and lets the kernel return.
// ---------------------------------------------------------------------------
constexpr unsigned long long kWaitNs = 2000000000ull;   // 2 s

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch. launch_dependents lets the next kernel in the
// stream be scheduled once every CTA of this grid has started; wait blocks
// until the previous grid in the stream has completed and its memory is
// visible (a no-op when this grid was launched without the attribute). Every
// kernel calls wait before its first global-memory access.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Streaming (evict-first) 16-byte global store.
__device__ __forceinline__ void st_stream_v4(void *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// ---------------------------------------------------------------------------
// cp.async (16 bytes, zero-filled when src_bytes == 0)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async_16(void *smem_dst, const void *gmem_src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem_dst)),
                 "l"(gmem_src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// alpha = fp32(scale_a * scale_w) from two device floats: the product of two
// floats is exact in double, rounded once to float.
__device__ __forceinline__ float alpha_from(const float *scales) {
    return __double2float_rn(__dmul_rn(static_cast<double>(scales[0]), static_cast<double>(scales[1])));
}

// The filter taps of a convolution that read input position `pos` along one
// axis: kk with pos + pad - kk*d = i*s for an output index 0 <= i < nout,
// listed as (tk[n], ti[n]); returns their number (at most k <= kMaxTapList).
// S = the stride when it is 1 or 2 (the divisions become shifts), 0 for any.
constexpr int kMaxTapList = 8;
template <int S>
__device__ __forceinline__ int tap_list(int pos, int pad, int k, int d, int s, int nout, int (&tk)[kMaxTapList],
                                        int (&ti)[kMaxTapList]) {
    int n = 0;
    for (int kk = 0; kk < k; ++kk) {
        const int r = pos + pad - kk * d;
        if (r < 0) break;                                     // r falls as kk grows
        int i;
        if constexpr (S == 1) {
            i = r;
        } else if constexpr (S == 2) {
            if (r & 1) continue;
            i = r >> 1;
        } else {
            if (r % s != 0) continue;
            i = r / s;
        }
        if (i < nout) { tk[n] = kk; ti[n] = i; ++n; }
    }
    return n;
}

}  // namespace bt
