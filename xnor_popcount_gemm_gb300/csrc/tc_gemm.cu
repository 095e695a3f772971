// Tensor-core contraction (tcgen05) over +1/-1 codes, for the linear layer
// and for the implicit-im2col convolution.
//
// The +1/-1 operands are stored as FP8 E4M3 or FP4 E2M1 codes (the pack
// kernel writes them); every product is +1 or -1, every partial sum an integer
// of magnitude <= K <= 16384, held exactly in the fp32 accumulator. So the
// accumulator is the integer dot = sum_k sa*sw = K - 2*hamming, and the
// epilogue applies y = fp32(dot * alpha) and the cast (bitorch-engine
// BinaryConv2dForward.forward: the native result scaled by
// scale_a*scale_w, then .to(x.dtype)). Zero codes (row padding, TMA zero fill
// outside the tensor, and taps that fall in a convolution's zero padding)
// contribute 0, which is the unfold + mm reading of padding.
//
// One CTA computes a 128 x 256 output tile with one tcgen05.mma chain
// (M=128, N=256, accumulator in 256 TMEM columns):
//   warp 0 lane 0   TMA producer: a ring of smem stages, each one 128- or
//                   64-byte-wide K slice of A (128 rows) and B (256 rows),
//                   written by TMA with the matching swizzle;
//   warp 1 lane 0   MMA issuer: 4 (or 2) MMAs of K = 32 bytes per stage,
//                   tcgen05.commit frees the stage;
//   warps 0..3      epilogue: tcgen05.ld of the warp's 32 TMEM lanes (rows),
//                   scale, cast, store.
// A convolution reads A through TMA im2col mode: for filter tap (kh, kw) the
// box is the 128 output pixels of the tile, each shifted by (kh*d, kw*d), the
// traversal stepping by the stride inside the padded bounding box.
#include <cudaTypedefs.h>

#include <mutex>

#include "bt_device.cuh"
#include "bt_internal.h"
#include "tc_ptx.cuh"

namespace bt {
namespace {

constexpr int kBM = 128, kBN = 256, kThreads = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol = 256;         // 32 columns of unit block scales (E2M1)
constexpr uint32_t kUnitScales = 0x7F7F7F7Fu;   // UE8M0 127 = 2^0 in every byte
constexpr int kSmemBudget = 200 * 1024;

struct TcArgs {
    int64_t M, N;
    int nk;                    // K steps (smem stages to consume)
    float alpha;
    void *out;
    unsigned int *err;
    // conv
    int Ho, Wo, s, p, d, k, cpt, rbc;
};

template <int ROWB> __host__ __device__ constexpr int stages_for() {
    return kSmemBudget / ((kBM + kBN) * ROWB) > 8 ? 8 : kSmemBudget / ((kBM + kBN) * ROWB);
}
template <int ROWB> __host__ __device__ constexpr int smem_bytes() {
    return stages_for<ROWB>() * (kBM + kBN) * ROWB + 1024 /*align*/ + 256 /*barriers*/;
}

template <int CODE, int ROWB>
__device__ __forceinline__ constexpr uint32_t instr_desc() {
    // D = F32, K-major A and B, N = 256, M = 128.
    return CODE == BT_CODE_E4M3
               ? ((1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t(kBN) >> 3) << 17) | ((uint32_t(kBM) >> 4) << 24))
               // block-scaled: A/B = E2M1, scale type UE8M0, scale-factor ids 0
               : ((1u << 7) | (1u << 10) | ((uint32_t(kBN) >> 3) << 17) | (1u << 23) |
                  ((uint32_t(kBM) >> 4) << 24));
}

template <int ROWB>
__device__ __forceinline__ uint64_t operand_desc(uint32_t saddr) {
    uint64_t d = tc::sw128_kmajor_desc(saddr);
    if (ROWB == 64) {
        // 64-byte swizzle: 8-row groups 512 bytes apart
        d &= ~((static_cast<uint64_t>(0x3FFF) << 32) | (static_cast<uint64_t>(7) << 61));
        d |= (static_cast<uint64_t>(512u >> 4) << 32) | (static_cast<uint64_t>(4u) << 61);
    }
    return d;
}

template <int OUT>
__device__ __forceinline__ void store_row_linear(typename OutT<OUT>::type *out, int64_t N, int64_t m, int64_t n,
                                                 const uint32_t (&r)[32], float alpha, bool vec_ok) {
    using T = typename OutT<OUT>::type;
    T v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = OutT<OUT>::cvt(__float2int_rn(__uint_as_float(r[j])), alpha);
    T *dst = out + m * N + n;
    if (vec_ok && n + 32 <= N) {
        constexpr int PER = 16 / sizeof(T);
#pragma unroll
        for (int q = 0; q < 32 / PER; ++q) *reinterpret_cast<uint4 *>(dst + q * PER) = *reinterpret_cast<const uint4 *>(&v[q * PER]);
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (n + j < N) dst[j] = v[j];
    }
}

template <int CODE, int ROWB, bool CONV, int OUT>
__global__ void __launch_bounds__(kThreads, 1)
tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const TcArgs a) {
    constexpr int S = stages_for<ROWB>();
    constexpr uint32_t kABytes = kBM * ROWB, kBBytes = kBN * ROWB;
    constexpr int kMmaPerStage = ROWB / 32;        // K = 32 bytes per MMA

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sA = base, sB = base + S * kABytes;
    const uint32_t bars = sB + S * kBBytes;               // full[S], empty[S], accum
    uint8_t *gbars = smem_raw + (bars - raw);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(gbars + 8 * (2 * S + 1));
    volatile uint32_t *abort_flag = tmem_slot + 1;
    auto full = [&](int s) { return bars + 8u * s; };
    auto empty = [&](int s) { return bars + 8u * (S + s); };
    const uint32_t accum = bars + 8u * (2 * S);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kBM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kBN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            tc::mbar_init(full(s), 1);
            tc::mbar_init(empty(s), 1);
        }
        tc::mbar_init(accum, 1);
        *abort_flag = 0u;
        tc::fence_mbar_init();
        tc::prefetch_map(&tmA);
        tc::prefetch_map(&tmB);
    }
    if (warp == 1) {
        tc::tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

    if (CODE == BT_CODE_E2M1) {
        // unit block scales for A and B: every byte of columns [256, 288)
        tc::tmem_st16_fill(tmem + lane_base + kSfCol, kUnitScales);
        tc::tmem_st16_fill(tmem + lane_base + kSfCol + 16, kUnitScales);
        tc::tmem_st_wait();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
    }

    // conv: base coordinates of the tile's first output pixel
    int cb = 0, ch = 0, cw = 0;
    if (CONV) {
        const int64_t hw = static_cast<int64_t>(a.Ho) * a.Wo;
        cb = static_cast<int>(m0 / hw);
        const int r = static_cast<int>(m0 - static_cast<int64_t>(cb) * hw);
        ch = (r / a.Wo) * a.s - a.p;
        cw = (r % a.Wo) * a.s - a.p;
    }

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int last_issue[8];
#pragma unroll
            for (int s = 0; s < 8; ++s) last_issue[s] = -1;
            bool ok = true;
            for (int kb = 0; kb < a.nk && ok; ++kb) {
                const int s = kb % S;
                const uint32_t ph = static_cast<uint32_t>(kb / S) & 1u;
                if (!tc::wait_bounded(empty(s), ph ^ 1u, abort_flag, a.err)) { ok = false; break; }
                tc::mbar_arrive_expect_tx(full(s), kABytes + kBBytes);
                if (CONV) {
                    const int tap = kb / a.cpt, chunk = kb - tap * a.cpt;
                    const int kh = tap / a.k, kw = tap - kh * a.k;
                    tc::tma_load_im2col_4d(sA + s * kABytes, &tmA, chunk * ROWB, cw, ch, cb,
                                           static_cast<uint16_t>(kw * a.d), static_cast<uint16_t>(kh * a.d), full(s));
                    tc::tma_load_2d(sB + s * kBBytes, &tmB, tap * a.rbc + chunk * ROWB, static_cast<int>(n0), full(s));
                } else {
                    tc::tma_load_2d(sA + s * kABytes, &tmA, kb * ROWB, static_cast<int>(m0), full(s));
                    tc::tma_load_2d(sB + s * kBBytes, &tmB, kb * ROWB, static_cast<int>(n0), full(s));
                }
                last_issue[s < 8 ? s : 0] = kb;
            }
            if (!ok) {
                // drain: let every issued copy land before the CTA can exit
                for (int s = 0; s < S && s < 8; ++s) {
                    if (last_issue[s] >= 0) {
                        const uint32_t ph = static_cast<uint32_t>(last_issue[s] / S) & 1u;
                        const unsigned long long t0 = globaltimer_ns();
                        while (!tc::mbar_try_wait(full(s), ph) && globaltimer_ns() - t0 < kWaitNs) {}
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t idesc = instr_desc<CODE, ROWB>();
            bool issued = false;
            for (int kb = 0; kb < a.nk; ++kb) {
                const int s = kb % S;
                const uint32_t ph = static_cast<uint32_t>(kb / S) & 1u;
                if (!tc::wait_bounded(full(s), ph, abort_flag, a.err)) break;
                tc::fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < kMmaPerStage; ++kk) {
                    const uint64_t ad = operand_desc<ROWB>(sA + s * kABytes + kk * 32);
                    const uint64_t bd = operand_desc<ROWB>(sB + s * kBBytes + kk * 32);
                    const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
                    if (CODE == BT_CODE_E4M3) tc::mma_f8f6f4(tmem, ad, bd, idesc, acc);
                    else tc::mma_mxf4(tmem, ad, bd, idesc, tmem + kSfCol, tmem + kSfCol + 16, acc);
                }
                issued = true;
                tc::mma_commit(empty(s));
            }
            // signals the epilogue (also when nothing was issued, so nobody waits in vain)
            (void)issued;
            tc::mma_commit(accum);
        }
        __syncwarp();
    }

    // ---------------- epilogue (all 4 warps) ----------------
    const bool have = tc::wait_bounded(accum, 0u, abort_flag, a.err);
    tc::fence_after_sync();
    if (have && *abort_flag == 0u) {
        using T = typename OutT<OUT>::type;
        T *out = static_cast<T *>(a.out);
        const int64_t m = m0 + warp * 32 + lane;
        const bool row_ok = m < a.M;
        const bool vec_ok = ((a.N * static_cast<int64_t>(sizeof(T))) % 16) == 0;
        int64_t ob = 0, pix = 0, hw = 0;
        if (CONV) {
            hw = static_cast<int64_t>(a.Ho) * a.Wo;
            ob = row_ok ? m / hw : 0;
            pix = m - ob * hw;
        }
#pragma unroll 1
        for (int c = 0; c < kBN; c += 32) {
            if (n0 + c >= a.N) break;                    // warp-uniform
            uint32_t r[32];
            tc::tmem_ld32(tmem + lane_base + static_cast<uint32_t>(c), r);
            tc::tmem_ld_wait();
            if (!row_ok) continue;
            if (CONV) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int64_t o = n0 + c + j;
                    if (o < a.N)
                        out[(ob * a.N + o) * hw + pix] = OutT<OUT>::cvt(__float2int_rn(__uint_as_float(r[j])), a.alpha);
                }
            } else {
                store_row_linear<OUT>(out, a.N, m, n0 + c, r, a.alpha, vec_ok);
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

PFN_cuTensorMapEncodeIm2col_v12000 encode_im2col() {
    static PFN_cuTensorMapEncodeIm2col_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeIm2col_v12000>(p);
    });
    return fn;
}

// 2-D byte matrix [rows, row_bytes] with row pitch `pitch`; box = box_inner bytes x box_rows.
bool map_2d(CUtensorMap *m, const void *ptr, uint64_t row_bytes, uint64_t pitch, uint64_t rows, uint32_t box_inner,
            uint32_t box_rows) {
    auto fn = encode_tiled();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {row_bytes, rows};
    cuuint64_t strides[1] = {pitch};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = box_inner == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int CODE, int ROWB, bool CONV, int OUT>
cudaError_t launch_t(const CUtensorMap &ma, const CUtensorMap &mb, const TcArgs &a, cudaStream_t s) {
    auto kern = tc_kernel<CODE, ROWB, CONV, OUT>;
    constexpr int smem = smem_bytes<ROWB>();
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] { attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); });
    if (attr_err != cudaSuccess) return attr_err;
    dim3 grid(static_cast<unsigned>((a.N + kBN - 1) / kBN), static_cast<unsigned>((a.M + kBM - 1) / kBM));
    kern<<<grid, kThreads, smem, s>>>(ma, mb, a);
    return cudaGetLastError();
}

template <int CODE, int ROWB, bool CONV>
cudaError_t launch_out(const CUtensorMap &ma, const CUtensorMap &mb, const TcArgs &a, bt_dtype out_t, cudaStream_t s) {
    switch (out_t) {
        case BT_F32: return launch_t<CODE, ROWB, CONV, BT_F32>(ma, mb, a, s);
        case BT_BF16: return launch_t<CODE, ROWB, CONV, BT_BF16>(ma, mb, a, s);
        case BT_F16: return launch_t<CODE, ROWB, CONV, BT_F16>(ma, mb, a, s);
        default: return launch_t<CODE, ROWB, CONV, BT_I32>(ma, mb, a, s);
    }
}

template <bool CONV>
cudaError_t launch_code(bt_code code, int rowb, const CUtensorMap &ma, const CUtensorMap &mb, const TcArgs &a,
                        bt_dtype out_t, cudaStream_t s) {
    if (code == BT_CODE_E4M3)
        return rowb == 128 ? launch_out<BT_CODE_E4M3, 128, CONV>(ma, mb, a, out_t, s)
                           : launch_out<BT_CODE_E4M3, 64, CONV>(ma, mb, a, out_t, s);
    return rowb == 128 ? launch_out<BT_CODE_E2M1, 128, CONV>(ma, mb, a, out_t, s)
                       : launch_out<BT_CODE_E2M1, 64, CONV>(ma, mb, a, out_t, s);
}

}  // namespace

bool tc_available() { return encode_tiled() != nullptr && encode_im2col() != nullptr; }

cudaError_t launch_tc_linear(const uint8_t *xp, const uint8_t *wp, bt_code code, int64_t M, int64_t N, int64_t K,
                             float alpha, void *out, bt_dtype out_t, unsigned int *err, cudaStream_t s) {
    const int64_t rb = row_bytes(K, code);
    CUtensorMap ma, mb;
    if (!map_2d(&ma, xp, rb, rb, M, 128, kBM) || !map_2d(&mb, wp, rb, rb, N, 128, kBN)) return cudaErrorInvalidValue;
    TcArgs a{};
    a.M = M; a.N = N; a.nk = static_cast<int>((rb + 127) / 128); a.alpha = alpha; a.out = out; a.err = err;
    return launch_code<false>(code, 128, ma, mb, a, out_t, s);
}

cudaError_t launch_tc_conv(const uint8_t *xp, const uint8_t *wp, bt_code code, const ConvGeom &g, float alpha,
                           void *out, bt_dtype out_t, unsigned int *err, cudaStream_t s) {
    const int64_t rbc = row_bytes(g.C, code);
    const int rowb = (rbc % 128 == 0) ? 128 : 64;
    auto fn = encode_im2col();
    if (fn == nullptr || rbc % 64 != 0) return cudaErrorInvalidValue;
    CUtensorMap ma, mb;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(rbc), static_cast<cuuint64_t>(g.W), static_cast<cuuint64_t>(g.H),
                          static_cast<cuuint64_t>(g.B)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(rbc), static_cast<cuuint64_t>(rbc * g.W),
                             static_cast<cuuint64_t>(rbc * g.W * g.H)};
    const int lo = -g.p, hi = g.p - (g.k - 1) * g.d;
    int lower[2] = {lo, lo}, upper[2] = {hi, hi};
    cuuint32_t estr[4] = {1, static_cast<cuuint32_t>(g.s), static_cast<cuuint32_t>(g.s), 1};
    const CUtensorMapSwizzle sw = rowb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (fn(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t *>(xp), dims, strides, lower, upper,
           static_cast<cuuint32_t>(rowb), kBM, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int64_t krow = static_cast<int64_t>(g.k) * g.k * rbc;
    if (!map_2d(&mb, wp, krow, krow, g.O, static_cast<uint32_t>(rowb), kBN)) return cudaErrorInvalidValue;
    TcArgs a{};
    a.M = g.B * g.Ho * g.Wo; a.N = g.O; a.alpha = alpha; a.out = out; a.err = err;
    a.Ho = static_cast<int>(g.Ho); a.Wo = static_cast<int>(g.Wo);
    a.s = g.s; a.p = g.p; a.d = g.d; a.k = g.k;
    a.cpt = static_cast<int>(rbc / rowb); a.rbc = static_cast<int>(rbc);
    a.nk = g.k * g.k * a.cpt;
    return launch_code<true>(code, rowb, ma, mb, a, out_t, s);
}

}  // namespace bt
