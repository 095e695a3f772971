// Tensor-core contraction (tcgen05) over +1/-1 codes, for the linear layer
// and for the convolution lowered to im2col rows.
//
// The +1/-1 operands are stored as FP8 E4M3 or FP4 E2M1 codes (the pack
// kernel writes them); every product is +1 or -1, every partial sum an integer
// of magnitude <= K <= 16384, held exactly in the fp32 accumulator. So the
// accumulator is the integer dot = sum_k sa*sw = K - 2*hamming, and the
// epilogue applies y = fp32(dot * alpha) and the cast (bitorch-engine
// BinaryConv2dForward.forward: the native result scaled by
// scale_a*scale_w, then .to(x.dtype)). Zero codes (row padding, TMA zero fill
// outside the tensor, and the zero taps the im2col rows hold for a
// convolution's padding) contribute 0, which is the unfold + mm reading of
// padding.
//
// D[r, c] = sum_k A[r, k] * B[c, k]: A and B are packed rows (K-major), read
// in 128-byte K slices. A linear layer has A = activations, B = weights and a
// row-major output [M, N]. A convolution has A = weights [O, k*k*C] and B =
// im2col rows [B*Ho*Wo, k*k*C], so a tile's rows are output channels and its
// columns output pixels: each TMEM lane holds a run of consecutive pixels of
// one channel, which is what the NCHW output wants.
//
// Persistent and warp-specialised, one CTA per SM. Two shapes:
//   single  a CTA computes 128 x BN tiles with cta_group::1 MMAs;
//   pair    a cluster of 2 CTAs computes 256 x BN tiles with cta_group::2
//           MMAs: each CTA loads its own 128 rows of A and half of the tile's
//           B rows, the even CTA issues the MMAs, and each CTA's TMEM holds
//           its 128 rows of the accumulator. Every SM receives 128 + BN/2
//           rows per K slice instead of 128 + BN, for the same MMA work.
// A smem stage holds D consecutive 128-byte K slices of A and of B, each
// operand loaded with one TMA box over a 3-D view {128 B, rows, slices} of
// its rows: on GB300 a TMA box costs a roughly fixed ~470 clocks of the SM's
// copy engine whatever its size, so two slices per box halve the cost per
// byte. A stage that reaches the row's last, partial slice is loaded slice by
// slice from the 2-D view instead, whose zero fill covers the half slice.
// The fp32 accumulator is double-buffered in TMEM (2 x 240 columns plus 32 of
// unit block scales for E2M1, 2 x 256 for E4M3), so a tile's epilogue -- and
// its output stores -- overlap the next tile's MMAs.
//   warp 0 lane 0   TMA producer: a ring of smem stages (128-byte swizzle),
//                   running ahead across tile boundaries.
//   warp 1 lane 0   MMA issuer (the even CTA of a pair): per 32 bytes of K
//                   one tcgen05.mma into the tile's accumulator buffer;
//                   tcgen05.commit frees the stage and, after a tile's last
//                   stage, hands the buffer to the epilogue.
//   warps 2..9      epilogue, two warps per TMEM lane quarter (32 rows) taking
//                   alternate 32-column boxes: the next box's TMEM load in
//                   flight while the current one is scaled, cast, and written
//                   to the warp's swizzled 32 x 32 smem box, from which whole
//                   row segments leave in 16-byte stores (or, for NCHW, runs
//                   of pixels in the widest aligned stores). Once both CTAs'
//                   warps have drained it, the buffer goes back to the MMA warp.
// Every wait is bounded (bt_set_wait_timeout, 2 s by default; the teardown's
// drains of copies and MMAs in flight always 2 s): a wait that runs out
// records BT_ERR_TIMEOUT in the device error word and the kernel winds down
// without trapping.
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <map>
#include <mutex>

#include "bt_device.cuh"
#include "bt_internal.h"
#include "tc_ptx.cuh"

namespace bt {
namespace {

constexpr int kBM = 128;                         // rows of A per CTA (= MMA M per CTA)
constexpr int kRowB = 128;                       // bytes of a K slice
constexpr int kEpiWarps = 8;                     // at most two per TMEM lane quarter
constexpr int kThreads = 64 + 32 * kEpiWarps;    // producer, MMA, epilogue warps (the most a launch takes)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol = 480;                 // 32 columns of unit block scales (E2M1)
constexpr uint32_t kUnitScales = 0x7F7F7F7Fu;    // UE8M0 127 = 2^0 in every byte
constexpr int kSmemMax = 232448;                 // 227 KB opt-in per CTA
// One staging box per epilogue warp: 32 rows x 32 outputs (4 KB for 4-byte
// outputs, 2 KB for 2-byte ones).
// Epilogue staging: one 32 x 32 box of outputs per epilogue warp.
__host__ __device__ constexpr int staging_bytes(int out_elem, int epi_warps = kEpiWarps) {
    return epi_warps * 32 * 32 * out_elem;
}
constexpr int kReserve = 1024 /*alignment*/ + 256 /*barriers*/;
constexpr int kMaxStages = 8;

// Output layouts: row-major; NCHW (convolution); row-major times the
// straight-through mask of x (bf16 or f32 x), for the backward's input gradient.
enum Layout { kRowsOut = 0, kNchwOut = 1, kRowsMaskBf16 = 2, kRowsMaskF32 = 3 };

struct TcArgs {
    int64_t M, N;              // D is M x N
    int slices;                // 128-byte K slices per row (the last may be half zero fill)
    int full_slices;           // whole slices: those the 3-D view covers
    int d;                     // K slices per smem stage
    int nk;                    // stages per tile
    int num_n, bn;             // column tiles; tile width BN (multiple of 16)
    int num_super;             // units of work: tiles (pairs: 256-row tiles) x K splits
    int num_tiles;             // tiles of one K split
    int64_t split_out;         // split-K: output elements between the splits' partial results
    uint32_t idesc;            // instruction descriptor
    float alpha;
    const float *scales;       // not null: alpha = fp32(scales[0] * scales[1]), read by the epilogue
    void *out;
    unsigned int *err;
    unsigned long long wait_ns;  // limit of each bounded wait of the main loops (teardown drains: kWaitNs)
    int vec;                   // rows: 1 when output rows are 16-byte aligned (16-byte stores)
                               // NCHW: bytes each lane stores at once (a run of one channel's pixels)
    int64_t hw;                // NCHW: output pixels per image (Ho * Wo)
    int stages;                // smem ring depth
    int epi_warps;             // epilogue warps of this launch: 4 (one per TMEM lane quarter) or 8 (two)
    const void *aux;           // masked layouts: x [M, N]
    float aux_scale;           // masked layouts: scale_a
    float aux_norm;            // masked layouts: 1 / sqrt(numel(x)), fp32
    float *aux_sum;            // masked layouts: sum(D * sign(x) * norm) accumulates here
};

// B rows one CTA holds per slice.
__host__ __device__ __forceinline__ int b_slot_rows(int bn, bool pair) { return pair ? bn / 2 : bn; }

// Shared memory: S stages of D slices of A (128 rows) and B, the epilogue
// staging boxes, barriers. S is as many stages as fit (at most 8).
int stage_bytes(int bn, bool pair, int d) { return (kBM + b_slot_rows(bn, pair)) * kRowB * d; }
int num_stages(int bn, bool pair, int d, int out_elem, int epi_warps = kEpiWarps) {
    const int s = (kSmemMax - kReserve - staging_bytes(out_elem, epi_warps)) / stage_bytes(bn, pair, d);
    return s > kMaxStages ? kMaxStages : s;
}
int smem_bytes(int bn, bool pair, int d, int out_elem, int epi_warps = kEpiWarps) {
    return num_stages(bn, pair, d, out_elem, epi_warps) * stage_bytes(bn, pair, d) + staging_bytes(out_elem, epi_warps) +
           kReserve;
}

// TMEM column of the second accumulator buffer; also the largest BN.
template <int CODE> __host__ __device__ constexpr uint32_t acc_stride() { return CODE == BT_CODE_E2M1 ? 240u : 256u; }

// Instruction descriptor: D = F32, K-major A and B, M rows (128, or 256 for a
// pair), N = bn.
uint32_t make_idesc(int code, int m, int bn) {
    const uint32_t mn = ((static_cast<uint32_t>(bn) >> 3) << 17) | ((static_cast<uint32_t>(m) >> 4) << 24);
    if (code == kCodeBF16) return (1u << 4) | (1u << 7) | (1u << 10) | mn;          // BF16 x BF16 -> F32
    if (code == BT_CODE_E4M3) return (1u << 4) | (0u << 7) | (0u << 10) | mn;       // E4M3 x E4M3
    return (1u << 7) | (1u << 10) | (1u << 23) | mn;   // block-scaled E2M1 x E2M1, UE8M0 scales, ids 0
}

// 16 bytes of converted outputs from accumulators r[j0 .. j0 + 16/elem).
template <int OUT, int ELEM>
__device__ __forceinline__ uint4 chunk16(const uint32_t (&r)[32], int j0, float alpha) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (ELEM == 4) {
            w[i] = FromAcc<OUT>::bits(__uint_as_float(r[j0 + i]), alpha);
        } else {
            w[i] = pack2_from_acc<OUT>(__uint_as_float(r[j0 + 2 * i]), __uint_as_float(r[j0 + 2 * i + 1]), alpha);
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Position of 16-byte chunk q of staging-box row `row`: the 128-byte swizzle
// (q ^ row % 8) for 4-byte outputs (128-byte rows), the 64-byte swizzle
// (q ^ (row / 2) % 4) for 2-byte outputs (64-byte rows), so that 32 lanes
// writing their rows' chunk q hit different banks.
template <int ELEM>
__device__ __forceinline__ uint32_t box_chunk(int q, int row) {
    return ELEM == 4 ? static_cast<uint32_t>(q ^ (row & 7)) : static_cast<uint32_t>(q ^ ((row >> 1) & 3));
}

// Global stores of 16, 8, 4 or 2 bytes (explicitly global; the low words of v).
template <int V> __device__ __forceinline__ void st_global(uint8_t *p, const uint4 &v) {
    if constexpr (V == 16)
        asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
    else if constexpr (V == 8)
        asm volatile("st.global.v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
    else if constexpr (V == 4)
        asm volatile("st.global.b32 [%0], %1;" ::"l"(p), "r"(v.x) : "memory");
    else
        asm volatile("st.global.b16 [%0], %1;" ::"l"(p), "h"(static_cast<uint16_t>(v.x)) : "memory");
}
template <int V> __device__ __forceinline__ uint4 ld_shared(uint32_t a) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if constexpr (V == 16)
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    else if constexpr (V == 8)
        asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    else if constexpr (V == 4)
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v.x) : "r"(a));
    else {
        uint16_t h;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(a));
        v.x = h;
    }
    return v;
}

// NCHW read-back of one staged 32 x 32 box (rows = channels, columns =
// pixels): each lane takes a run of V bytes (V / ELEM consecutive pixels,
// inside one image and V-aligned) of one channel row; 32 / LPR rows per
// instruction, so each store instruction covers whole runs of several rows.
// `col` is the box's first column (pixel), `row0` its first row.
template <int V, int ELEM>
__device__ __forceinline__ void nchw_box(uint8_t *out, uint32_t sbox, int lane, uint32_t col, uint32_t ncol_end,
                                         int64_t row0, int64_t M, uint32_t hw) {
    constexpr int kBoxRow = 32 * ELEM;
    constexpr int kLpr = kBoxRow / V;                    // lanes per row
    constexpr int kRowsPer = 32 / kLpr;
    const int q = lane % kLpr;
    const uint32_t c = col + static_cast<uint32_t>(q * (V / ELEM));
    if (c >= ncol_end) return;
    const uint32_t ob = c / hw, pix = c - ob * hw;
    uint8_t *base = out + (static_cast<int64_t>(ob) * M * hw + pix) * ELEM;
    const uint32_t qb = static_cast<uint32_t>(q * V);
    // all shared-memory reads first, then all stores (the asm statements keep
    // their order, so interleaving them would expose each read's latency)
    constexpr int kIters = 32 / kRowsPer;
    uint4 v[kIters];
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
        const int rr = lane / kLpr + i * kRowsPer;
        v[i] = ld_shared<V>(sbox + static_cast<uint32_t>(rr * kBoxRow) +
                            (box_chunk<ELEM>(static_cast<int>(qb >> 4), rr) << 4) + (qb & 15u));
    }
    const int64_t plane = static_cast<int64_t>(hw) * ELEM;
    uint8_t *p = base + (row0 + lane / kLpr) * plane;
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
        if (row0 + lane / kLpr + i * kRowsPer >= M) break;
        st_global<V>(p + static_cast<int64_t>(i * kRowsPer) * plane, v[i]);
    }
}

// One 16-byte chunk of eight bf16 outputs y at x[idx .. idx + 8): each
// becomes y * middle, middle = !(q < -1 || q > 1) for q = x / scale_a in x's
// dtype, and sum(y * middle * sign(x) * norm) (each product rounded to fp32)
// is added to tsum. sign(x) = (x > 0) - (x < 0).
// Whether q = x / scale_a (fp32 division, then rounded to bf16 for a bf16 x)
// lies outside [-1, 1]. x * (1 / scale_a) is within a few ulps of x / scale_a,
// so it decides every x whose quotient is not near the boundary (1 for an
// f32 x; 1 + 2^-8, the point where bf16 rounding leaves 1, for a bf16 x); the
// rest take the division.
template <bool BF16X>
__device__ __forceinline__ bool outside_unit(float x, float scale_a, float inv_scale) {
    constexpr float kEdge = BF16X ? 1.00390625f : 1.0f;
    const float qa = fabsf(x * inv_scale);
    if (qa < kEdge * 0.99999f) return false;
    if (qa > kEdge * 1.00001f) return true;
    float q = __fdiv_rn(x, scale_a);
    if constexpr (BF16X) q = __bfloat162float(__float2bfloat16_rn(q));
    return q < -1.0f || q > 1.0f;
}

// Eight consecutive elements of x (bf16 or f32), loaded ahead of their use.
template <int LAYOUT> struct XChunk {
    uint4 a, b;
    __device__ __forceinline__ void load(const void *x, int64_t idx) {
        if constexpr (LAYOUT == kRowsMaskBf16) {
            a = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(x) + idx));
        } else {
            a = __ldg(reinterpret_cast<const uint4 *>(static_cast<const float *>(x) + idx));
            b = __ldg(reinterpret_cast<const uint4 *>(static_cast<const float *>(x) + idx + 4));
        }
    }
    __device__ __forceinline__ void to_f32(float (&xf)[8]) const {
        if constexpr (LAYOUT == kRowsMaskBf16) {
            const uint32_t xw[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) xf[e] = __uint_as_float(((xw[e >> 1] >> (16 * (e & 1))) & 0xFFFFu) << 16);
        } else {
            const uint32_t xw[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) xf[e] = __uint_as_float(xw[e]);
        }
    }
};

template <int LAYOUT>
__device__ __forceinline__ uint4 mask_chunk(const uint4 &v, const XChunk<LAYOUT> &xc, float scale_a, float norm,
                                            float &tsum) {
    float xf[8];
    xc.to_f32(xf);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const float inv_scale = 1.0f / scale_a;
    uint32_t o[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float y = __uint_as_float(((w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu) << 16);
        const bool out = outside_unit<LAYOUT == kRowsMaskBf16>(xf[e], scale_a, inv_scale);
        const float ym = __fmul_rn(y, out ? 0.0f : 1.0f);
        const float sg = (xf[e] > 0.0f ? 1.0f : 0.0f) - (xf[e] < 0.0f ? 1.0f : 0.0f);
        tsum = __fadd_rn(tsum, __fmul_rn(__fmul_rn(ym, sg), norm));
        o[e >> 1] |= (__float_as_uint(ym) >> 16) << (16 * (e & 1));        // ym is y or +-0: exact in bf16
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int CODE, int LAYOUT, int OUT, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
tc_kernel(const __grid_constant__ CUtensorMap tmA3, const __grid_constant__ CUtensorMap tmB3,
          const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2, const TcArgs a) {
    constexpr uint32_t kASlice = kBM * kRowB;      // A bytes per K slice (128 rows)
    constexpr int kMmaPerSlice = kRowB / 32;       // K = 32 bytes per MMA
    using T = typename OutT<OUT>::type;
    constexpr int kElem = sizeof(T);
    constexpr int kBoxInner = 32 * kElem;          // bytes of one staging-box row: 32 output columns
    constexpr int kTileRows = PAIR ? 2 * kBM : kBM;
    const int S = a.stages;
    const int bn = a.bn;
    const int D = a.d;
    const uint32_t kBSlice = static_cast<uint32_t>(b_slot_rows(bn, PAIR) * kRowB);   // B bytes per K slice
    const uint32_t kAStage = kASlice * D, kBStage = kBSlice * D;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sA = base, sB = base + S * kAStage;
    const uint32_t sStage = sB + S * kBStage;                        // epilogue staging boxes
    const uint32_t bars = sStage + staging_bytes(kElem, a.epi_warps);   // full[S], empty[S], tfull[2], tempty[2], drain
    uint8_t *gbars = smem_raw + (bars - raw);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(gbars + 8 * (2 * kMaxStages + 5));
    volatile uint32_t *abort_flag = tmem_slot + 1;
    auto full = [&](int s) { return bars + 8u * s; };
    auto empty = [&](int s) { return bars + 8u * (kMaxStages + s); };
    auto tfull = [&](int b) { return bars + 8u * (2 * kMaxStages + b); };      // accumulator buffer b written
    auto tempty = [&](int b) { return bars + 8u * (2 * kMaxStages + 2 + b); }; // accumulator buffer b drained
    const uint32_t drain = bars + 8u * (2 * kMaxStages + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = PAIR ? tc::cluster_ctarank() : 0u;
    const bool leader = !PAIR || crank == 0;                         // issues the MMAs

    if (threadIdx.x == 0) pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            tc::mbar_init(full(s), 1);
            tc::mbar_init(empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(tfull(b), 1);
            // one arrival per epilogue warp (of both CTAs of a pair)
            tc::mbar_init(tempty(b), static_cast<uint32_t>(PAIR ? 2 * a.epi_warps : a.epi_warps));
        }
        tc::mbar_init(drain, 1);
        *abort_flag = 0u;
        tc::fence_mbar_init();
        tc::prefetch_map(&tmA3);
        tc::prefetch_map(&tmB3);
        tc::prefetch_map(&tmA2);
        tc::prefetch_map(&tmB2);
    }
    if (warp == 1) {
        if (PAIR) {
            tc::tmem_alloc_pair(smem_u32(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
            tc::tmem_relinquish_pair();
        } else {
            tc::tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
            tc::tmem_relinquish();
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int quarter = warp & 3;                                   // TMEM lanes this warp may touch
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    if (CODE == BT_CODE_E2M1 && warp >= 2 && warp < 6) {
        // unit block scales for A and B: every byte of the last 32 columns
        tc::tmem_st16_fill(tmem + lane_base + kSfCol, kUnitScales);
        tc::tmem_st16_fill(tmem + lane_base + kSfCol + 16, kUnitScales);
        tc::tmem_st_wait();
    }
    tc::fence_before_sync();
    __syncthreads();
    // the peer's barriers and block scales exist before any copy, commit or MMA reaches them
    if (PAIR) tc::cluster_sync();
    tc::fence_after_sync();

    const int unit = PAIR ? static_cast<int>(tc::cluster_id_x()) : static_cast<int>(blockIdx.x);
    const int nunits = PAIR ? static_cast<int>(tc::num_clusters_x()) : static_cast<int>(gridDim.x);
    // rows of the A tile and of the B tile this CTA loads
    const int a_first = PAIR ? static_cast<int>(crank) * kBM : 0;
    const int b_rows = b_slot_rows(bn, PAIR);
    const int b_first = PAIR ? static_cast<int>(crank) * b_rows : 0;
    // slices of stage kb of a tile: [kb * D, kb * D + count)
    auto slice_count = [&](int kb) { return a.slices - kb * D < D ? a.slices - kb * D : D; };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            pdl_wait();                                   // operands come from the previous kernel
            // a pair's copies complete on the even CTA's full barriers, which
            // expect the bytes of both CTAs
            const uint32_t slice_bytes = static_cast<uint32_t>((PAIR ? 2 : 1) * (kBM + b_rows) * kRowB);
            int s = 0;                                    // ring slot and its phase
            uint32_t ph = 0;
            uint32_t last_phase[kMaxStages];              // phase of each slot's last copy; 2 = none
#pragma unroll
            for (int i = 0; i < kMaxStages; ++i) last_phase[i] = 2u;
            bool ok = true;
            for (int st = unit; st < a.num_super && ok; st += nunits) {
                // K split `sp` covers slices [sp * slices, (sp + 1) * slices) of the rows
                const int sp = st / a.num_tiles, tl = st - sp * a.num_tiles;
                const int mt = tl / a.num_n, nt = tl % a.num_n;
                const int am0 = mt * kTileRows + a_first;
                const int bn0 = nt * bn + b_first;
                for (int kb = 0; kb < a.nk; ++kb) {
                    if (!tc::wait_fast(empty(s), ph ^ 1u, abort_flag, a.err, a.wait_ns)) { ok = false; break; }
                    const uint32_t adst = sA + s * kAStage, bdst = sB + s * kBStage;
                    const uint32_t fbar = PAIR ? tc::mapa(full(s), 0u) : full(s);
                    const int k0 = sp * a.slices + kb * D;
                    const bool whole = kb * D + D <= a.slices && k0 + D <= a.full_slices;
                    if (whole) {
                        // D whole slices: one box per operand
                        if (leader) tc::mbar_arrive_expect_tx(full(s), slice_bytes * D);
                        if (PAIR) {
                            tc::tma_load_3d_pair(adst, &tmA3, 0, am0, k0, fbar);
                            tc::tma_load_3d_pair(bdst, &tmB3, 0, bn0, k0, fbar);
                        } else {
                            tc::tma_load_3d(adst, &tmA3, 0, am0, k0, fbar);
                            tc::tma_load_3d(bdst, &tmB3, 0, bn0, k0, fbar);
                        }
                    } else {
                        // the row's last stage: slice by slice from the 2-D view
                        const int cnt = slice_count(kb);
                        if (leader) tc::mbar_arrive_expect_tx(full(s), slice_bytes * cnt);
                        for (int i = 0; i < cnt; ++i) {
                            const uint32_t ad = adst + i * kASlice, bd = bdst + i * kBSlice;
                            if (PAIR) {
                                tc::tma_load_2d_pair(ad, &tmA2, (k0 + i) * kRowB, am0, fbar);
                                tc::tma_load_2d_pair(bd, &tmB2, (k0 + i) * kRowB, bn0, fbar);
                            } else {
                                tc::tma_load_2d(ad, &tmA2, (k0 + i) * kRowB, am0, fbar);
                                tc::tma_load_2d(bd, &tmB2, (k0 + i) * kRowB, bn0, fbar);
                            }
                        }
                    }
                    last_phase[s] = ph;
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok && leader) {
                // let every issued copy land before the CTA can exit (a pair's
                // copies all complete on the even CTA's barriers)
                for (int i = 0; i < S; ++i) {
                    if (last_phase[i] < 2u) {
                        const unsigned long long t0 = globaltimer_ns();
                        while (!tc::mbar_try_wait(full(i), last_phase[i]) && globaltimer_ns() - t0 < kWaitNs) {}
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer ----------------
            int s = 0;
            uint32_t ph = 0;
            int local = 0;
            bool ok = true;
            for (int st = unit; st < a.num_super && ok; st += nunits, ++local) {
                const int buf = local & 1;
                if (local >= 2) {
                    // the epilogue (of both CTAs of a pair) has drained this buffer
                    if (!tc::wait_fast(tempty(buf), static_cast<uint32_t>((local - 2) >> 1) & 1u, abort_flag, a.err, a.wait_ns))
                        break;
                    tc::fence_after_sync();
                }
                const uint32_t dacc = tmem + static_cast<uint32_t>(buf) * acc_stride<CODE>();
                for (int kb = 0; kb < a.nk; ++kb) {
                    if (!tc::wait_fast(full(s), ph, abort_flag, a.err, a.wait_ns)) { ok = false; break; }
                    tc::fence_after_sync();
                    const int cnt = slice_count(kb);
                    // descriptors built per MMA from 32-bit addresses (measured on GB300:
                    // adding 64-bit offsets to descriptors built once per stage made the
                    // bf16 products of the backward ~6 % slower, the E2M1 forward no faster)
                    for (int i = 0; i < cnt; ++i) {
#pragma unroll
                        for (int kk = 0; kk < kMmaPerSlice; ++kk) {
                            const uint64_t ad = tc::sw128_kmajor_desc(sA + s * kAStage + i * kASlice + kk * 32);
                            const uint64_t bd = tc::sw128_kmajor_desc(sB + s * kBStage + i * kBSlice + kk * 32);
                            const uint32_t acc = (kb | i | kk) != 0 ? 1u : 0u;
                            if (PAIR) {
                                if (CODE == kCodeBF16) tc::mma_f16_pair(dacc, ad, bd, a.idesc, acc);
                                else if (CODE == BT_CODE_E4M3) tc::mma_f8f6f4_pair(dacc, ad, bd, a.idesc, acc);
                                else tc::mma_mxf4_pair(dacc, ad, bd, a.idesc, tmem + kSfCol, tmem + kSfCol + 16, acc);
                            } else {
                                if (CODE == kCodeBF16) tc::mma_f16(dacc, ad, bd, a.idesc, acc);
                                else if (CODE == BT_CODE_E4M3) tc::mma_f8f6f4(dacc, ad, bd, a.idesc, acc);
                                else tc::mma_mxf4(dacc, ad, bd, a.idesc, tmem + kSfCol, tmem + kSfCol + 16, acc);
                            }
                        }
                    }
                    if (PAIR) tc::mma_commit_pair(empty(s), 0x3);
                    else tc::mma_commit(empty(s));
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
                if (ok) {
                    if (PAIR) tc::mma_commit_pair(tfull(buf), 0x3);
                    else tc::mma_commit(tfull(buf));
                }
            }
            // every MMA issued must finish before the accumulator is freed
            if (PAIR) tc::mma_commit_pair(drain, 0x1);
            else tc::mma_commit(drain);
            const unsigned long long t0 = globaltimer_ns();
            while (!tc::mbar_try_wait(drain, 0u) && globaltimer_ns() - t0 < kWaitNs) {}
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (warps 2..9) ----------------
        pdl_wait();                                       // the previous kernel may still use `out`
        T *const out_base = static_cast<T *>(a.out);
        const uint32_t sbox = sStage + static_cast<uint32_t>((warp - 2) * 32 * kBoxInner);   // this warp's staging box
        constexpr bool kMask = LAYOUT == kRowsMaskBf16 || LAYOUT == kRowsMaskF32;
        const float alpha = a.scales != nullptr ? alpha_from(a.scales) : a.alpha;
        float tsum = 0.0f;                                // masked layouts: this lane's grad_scale_a terms
        int local = 0;
        for (int st = unit; st < a.num_super; st += nunits, ++local) {
            const int sp = st / a.num_tiles, tl = st - sp * a.num_tiles;
            const int mt = tl / a.num_n, nt = tl % a.num_n;
            T *const out = out_base + sp * a.split_out;           // split-K: this split's partial result
            const int64_t m0 = static_cast<int64_t>(mt) * kTileRows + (PAIR ? static_cast<int64_t>(crank) * kBM : 0);
            const int n0 = nt * bn;
            const int buf = local & 1;
            if (!tc::wait_fast(tfull(buf), static_cast<uint32_t>(local >> 1) & 1u, abort_flag, a.err, a.wait_ns)) break;
            tc::fence_after_sync();
            bool released = false;
            auto release = [&]() {
                // every TMEM read of this tile is complete: hand the accumulators back
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if (PAIR && crank != 0) tc::mbar_arrive_cluster(tc::mapa(tempty(buf), 0u));
                    else tc::mbar_arrive(tempty(buf));
                }
                released = true;
            };
            const int64_t ncols = a.N - n0 < bn ? a.N - n0 : bn;
            const int64_t ncol_end = n0 + ncols;                             // this tile's columns end here
            const int nbox = ncols > 0 ? static_cast<int>((ncols + 31) / 32) : 0;
            const int64_t mrow0 = m0 + quarter * 32;                         // this warp's first row
            // the two warps of a lane quarter take alternate 32-column boxes
            // the warps of a lane quarter take its 32-column boxes in turn
            const int wpq = a.epi_warps / 4, half = (warp - 2) / 4;
            const int total = mrow0 < a.M && nbox > half ? (nbox - half + wpq - 1) / wpq : 0;   // this warp's boxes
            const uint32_t tbase = tmem + lane_base + static_cast<uint32_t>(buf) * acc_stride<CODE>();
            auto tcol_of = [&](int j) { return tbase + static_cast<uint32_t>(32 * (wpq * j + half)); };
            auto emit = [&](const uint32_t (&r)[32], int j) {
                const int c0 = 32 * (wpq * j + half);
                // masked layouts: this lane's x chunks (the rows and columns of the
                // 16-byte chunks it stores below) go in flight before the staging
                XChunk<LAYOUT == kRowsMaskF32 ? kRowsMaskF32 : kRowsMaskBf16> xc[4];
                if constexpr (kMask) {
                    constexpr int kCh = kBoxInner / 16, kRp = 32 / kCh;
                    static_assert(32 / kRp <= 4, "x chunks per lane");
                    const int64_t xcol = n0 + c0 + (lane % kCh) * (16 / kElem), xrow = mrow0 + lane / kCh;
                    if (xcol < ncol_end) {
#pragma unroll
                        for (int i = 0; i < 32 / kRp; ++i)
                            if (xrow + i * kRp < a.M) xc[i].load(a.aux, (xrow + i * kRp) * a.N + xcol);
                    }
                }
                // stage the box: row = this lane's TMEM lane, 32 columns, swizzled;
                // reading it back across rows lets every store instruction cover
                // whole row segments
                __syncwarp();                                                 // previous box fully read back
                constexpr int kChunks = kBoxInner / 16;
#pragma unroll
                for (int q = 0; q < kChunks; ++q) {
                    const uint32_t addr = sbox + static_cast<uint32_t>(lane * kBoxInner) + (box_chunk<kElem>(q, lane) << 4);
                    const uint4 w = chunk16<OUT, kElem>(r, q * (16 / kElem), alpha);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w.x), "r"(w.y), "r"(w.z),
                                 "r"(w.w)
                                 : "memory");
                }
                __syncwarp();
                if constexpr (LAYOUT == kNchwOut) {
                    uint8_t *ob = reinterpret_cast<uint8_t *>(out);
                    const uint32_t col = static_cast<uint32_t>(n0 + c0), cend = static_cast<uint32_t>(ncol_end);
                    const uint32_t hw = static_cast<uint32_t>(a.hw);
                    if (a.vec == 16) nchw_box<16, kElem>(ob, sbox, lane, col, cend, mrow0, a.M, hw);
                    else if (a.vec == 8) nchw_box<8, kElem>(ob, sbox, lane, col, cend, mrow0, a.M, hw);
                    else if constexpr (kElem == 4) nchw_box<4, kElem>(ob, sbox, lane, col, cend, mrow0, a.M, hw);
                    else if (a.vec == 4) nchw_box<4, kElem>(ob, sbox, lane, col, cend, mrow0, a.M, hw);
                    else nchw_box<2, kElem>(ob, sbox, lane, col, cend, mrow0, a.M, hw);
                } else if (a.vec) {
                    // aligned rows: read the box back as 16-byte chunks, kChunks lanes
                    // per row, 32/kChunks rows per instruction, and store them whole
                    constexpr int kRowsPer = 32 / kChunks;
                    constexpr int kIters = 32 / kRowsPer;
                    const int q = lane % kChunks;
                    const int64_t col = n0 + c0 + q * (16 / kElem);
                    // all shared-memory reads first, then all stores
                    uint4 v[kIters];
#pragma unroll
                    for (int i = 0; i < kIters; ++i) {
                        const int rr = i * kRowsPer + lane / kChunks;
                        v[i] = ld_shared<16>(sbox + static_cast<uint32_t>(rr * kBoxInner) + (box_chunk<kElem>(q, rr) << 4));
                    }
                    if (col < ncol_end) {
                        const int64_t row = mrow0 + lane / kChunks;
                        uint8_t *p = reinterpret_cast<uint8_t *>(out) + (row * a.N + col) * kElem;
                        if constexpr (kMask) {
#pragma unroll
                            for (int i = 0; i < kIters; ++i)
                                if (row + i * kRowsPer < a.M)
                                    v[i] = mask_chunk<LAYOUT>(v[i], xc[i], a.aux_scale, a.aux_norm, tsum);
                        }
#pragma unroll
                        for (int i = 0; i < kIters; ++i)
                            if (row + i * kRowsPer < a.M)
                                st_stream_v4(p + static_cast<int64_t>(i * kRowsPer) * a.N * kElem, v[i]);
                    }
                } else if constexpr (!kMask) {
                    // ragged N: read the box back one row at a time, lanes along
                    // the columns, so every store is 32 consecutive elements
                    const int64_t col = n0 + c0 + lane;
                    constexpr int kPer = 16 / kElem;
                    const uint32_t off = static_cast<uint32_t>((lane % kPer) * kElem);
#pragma unroll 4
                    for (int rr = 0; rr < 32; ++rr) {
                        const uint32_t addr =
                            sbox + static_cast<uint32_t>(rr * kBoxInner) + (box_chunk<kElem>(lane / kPer, rr) << 4) + off;
                        uint32_t v;
                        if (kElem == 4) asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
                        else asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(addr));
                        const int64_t row = mrow0 + rr;
                        if (row < a.M && col < ncol_end) {
                            if (kElem == 4) reinterpret_cast<uint32_t *>(out)[row * a.N + col] = v;
                            else reinterpret_cast<uint16_t *>(out)[row * a.N + col] = static_cast<uint16_t>(v);
                        }
                    }
                }
            };
            uint32_t r0[32], r1[32];
            if (total > 0) tc::tmem_ld32(tcol_of(0), r0);
#pragma unroll 1
            for (int b = 0; b < total; b += 2) {
                tc::tmem_ld_wait();
                if (b + 1 < total) tc::tmem_ld32(tcol_of(b + 1), r1);
                else release();
                emit(r0, b);
                if (b + 1 < total) {
                    tc::tmem_ld_wait();
                    if (b + 2 < total) tc::tmem_ld32(tcol_of(b + 2), r0);
                    else release();
                    emit(r1, b + 1);
                }
            }
            if (!released) release();
        }
        if constexpr (kMask) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) tsum += __shfl_xor_sync(0xFFFFFFFFu, tsum, o);
            if (lane == 0) atomicAdd(a.aux_sum, tsum);
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    // no CTA of a pair leaves while its peer may still signal its barriers or
    // run MMAs on its shared memory and TMEM
    if (PAIR) tc::cluster_sync();
    if (warp == 1) {
        tc::fence_after_sync();
        if (PAIR) tc::tmem_dealloc_pair(tmem, kTmemCols);
        else tc::tmem_dealloc(tmem, kTmemCols);
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

int sm_count() { return device_sm_count(); }

// Views of a byte matrix [rows, row_bytes] (row pitch `pitch` >= row_bytes,
// both multiples of 16), 128-byte swizzle, zero fill outside:
//   2-D {row_bytes, rows}, box 128 bytes x box_rows;
//   3-D {128, rows, full slices} (strides pitch, 128), box 128 x box_rows x
//   d: d consecutive whole K slices in one copy, landing slice after slice.
bool map_2d(CUtensorMap *m, const void *ptr, uint64_t row_bytes, uint64_t pitch, uint64_t rows, uint32_t box_rows) {
    auto fn = encode_tiled();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {row_bytes, rows};
    cuuint64_t strides[1] = {pitch};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kRowB), box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool map_3d(CUtensorMap *m, const void *ptr, uint64_t pitch, uint64_t rows, uint64_t full_slices,
            uint32_t box_rows, uint32_t d) {
    auto fn = encode_tiled();
    if (fn == nullptr) return false;
    // rows without a whole slice never use this view: encode a one-row stand-in
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kRowB), full_slices > 0 ? rows : 1, full_slices > 0 ? full_slices : 1};
    cuuint64_t strides[2] = {full_slices > 0 ? pitch : static_cast<cuuint64_t>(kRowB), static_cast<cuuint64_t>(kRowB)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(kRowB), box_rows, d};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tile configuration: the shape (single CTAs or CTA pairs), BN (a multiple of
// 16 up to 240 for E2M1 / 256 for E4M3; the epilogue masks the part of its
// last 32-column box past the tile) and D, the K slices per stage.
// The cost model, whose constants are estimates fitted to measurements on
// GB300 (2070 MHz; standalone probes and timing-only copies of this kernel
// that are not part of this repository): a problem takes
// `rounds` waves of tiles over the SMs (pairs: SMs / 2 at a time). A K slice
// costs the largest of
//   - its MMA time: an M=128 MMA of 32 bytes of K per row takes N / 2 clocks
//     per SM, pair or not (4 MMAs per slice);
//   - the shared-memory traffic it puts on one SM, at about 125 bytes per
//     clock: the copies written (128 A rows and the B rows this SM loads)
//     plus the operand reads of the MMAs (128 A rows, and BN B rows: a pair's
//     B half is read by both SMs' tensor cores);
//   - its share of the copy engine: about 480 clocks per TMA box of up to two
//     slices, whatever its size (560 for four), two boxes per stage;
// plus about 1000 clocks per tile. The epilogue (about 20 clocks per output
// column of the CTA's 128 rows; 30 for a pair, whose tcgen05.ld of one buffer
// waits behind the pair MMAs writing the other) overlaps the next tile's MMAs
// and shows only where it is the longer of the two, and once for the last tile.
// BT_TC_CONFIG="bn,d" (single) or "pair,bn,d" overrides the choice.
struct TileCfg {
    bool pair;
    int bn, d;
    double cost;     // modelled clocks of the whole launch
};

double tile_cost(bool pair, int bn, int d, int64_t M, int64_t N, int slices, int sms, int splits) {
    const int rows = pair ? 2 * kBM : kBM;
    const int64_t num_m = (M + rows - 1) / rows, num_n = (N + bn - 1) / bn;
    const int64_t units = pair ? sms / 2 : sms;
    const int64_t tiles = num_m * num_n * splits;          // every K split of every tile is a unit of work
    const int64_t rounds = (tiles + units - 1) / units;
    const double mma = (kRowB / 32) * (bn / 2.0);
    const double written = static_cast<double>(kBM + b_slot_rows(bn, pair)) * kRowB;
    const double read = static_cast<double>(kBM + bn) * kRowB;
    const double smem = (written + read) / 125.0;
    const double copy = 2.0 * (d <= 2 ? 480.0 : 560.0) / d;
    double slice = mma > smem ? mma : smem;
    if (copy > slice) slice = copy;
    double tile = slices * slice + 1000.0;
    const double epi = (pair ? 30.0 : 20.0) * bn;
    if (epi > tile) tile = epi;
    return static_cast<double>(rounds) * tile + epi + 600.0;
}

bool valid_shape(bool pair, int bn, int d, int max_bn, int out_elem, int epi) {
    return bn >= 32 && bn <= max_bn && bn % 16 == 0 && d >= 1 && d <= 4 &&
           num_stages(bn, pair, d, out_elem, epi) >= 2;
}

// `pick` (a measured or forced shape, or nullptr) is taken when it is valid
// for this problem; the environment's BT_TC_CONFIG comes first.
TileCfg choose_cfg(int64_t M, int64_t N, int slices, int sms, int max_bn, int out_elem, int splits,
                   const TcTileChoice *pick = nullptr) {
    if (const char *env = std::getenv("BT_TC_CONFIG")) {
        int bn = 0, d = 0;
        const bool pair = std::strncmp(env, "pair,", 5) == 0;
        if (std::sscanf(pair ? env + 5 : env, "%d,%d", &bn, &d) == 2 && valid_shape(pair, bn, d, max_bn, out_elem, kEpiWarps))
            return TileCfg{pair, bn, d, 0.0};
    }
    if (pick != nullptr && valid_shape(pick->pair != 0, pick->bn, pick->d, max_bn, out_elem, pick->epi))
        return TileCfg{pick->pair != 0, pick->bn, pick->d, 0.0};
    TileCfg best{false, max_bn, 1, -1.0};
    for (int p = 1; p >= 0; --p)
        for (int d = 4; d >= 1; d /= 2)
            for (int bn = max_bn; bn >= 32; bn -= 16) {
                if (num_stages(bn, p == 1, d, out_elem) < 2) continue;
                const double c = tile_cost(p == 1, bn, d, M, N, slices, sms, splits);
                if (best.cost < 0.0 || c < best.cost * 0.999) best = TileCfg{p == 1, bn, d, c};
            }
    return best;
}

struct Maps {
    CUtensorMap a3, b3, a2, b2;
};

// Epilogue warps of a launch, and with them the staging (one 32 x 32 box per
// warp). The forward linears take one per TMEM lane quarter where each tile's
// output rows are 16-byte aligned (whole-chunk stores) and its main loop (>= 8
// K slices) hides the slower epilogue: the smaller staging keeps the CTA's
// shared memory under the next carveout step (measured on GB300, same box: the
// 8192x4096x11008 step 149 -> 141 us and the 4096^3 one 33.3 -> 31.5 us with
// four-warp staging, whether or not the launch bound changed; eight warps with
// eight-warp staging 148.8 / 32.9). Ragged rows (element stores) and the other
// layouts keep two per quarter (the ragged linear measured 90 us with two,
// 118 with one). BT_TC_EPI=4 or 8 in the environment forces either.
int epilogue_warps(int code, int layout, const TcArgs &a) {
    if (const char *env = std::getenv("BT_TC_EPI")) {
        if (std::strcmp(env, "4") == 0) return 4;
        if (std::strcmp(env, "8") == 0) return 8;
    }
    if (a.epi_warps == 4 || a.epi_warps == 8) return a.epi_warps;      // a measured or forced shape's count
    const bool forward = code == BT_CODE_E2M1 || code == BT_CODE_E4M3;
    return forward && layout == kRowsOut && a.vec && a.slices >= 8 ? 4 : 8;
}

template <int CODE, int LAYOUT, int OUT, bool PAIR>
cudaError_t launch_t(const Maps &mp, TcArgs a, cudaStream_t s) {
    auto kern = tc_kernel<CODE, LAYOUT, OUT, PAIR>;
    a.epi_warps = epilogue_warps(CODE, LAYOUT, a);
    a.stages = num_stages(a.bn, PAIR, a.d, static_cast<int>(sizeof(typename OutT<OUT>::type)), a.epi_warps);
    a.wait_ns = wait_limit_ns();
    const int smem = smem_bytes(a.bn, PAIR, a.d, static_cast<int>(sizeof(typename OutT<OUT>::type)), a.epi_warps);
    if (a.stages < 2 || smem > kSmemMax) return cudaErrorInvalidValue;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] { attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax); });
    if (attr_err != cudaSuccess) return attr_err;
    const int csize = PAIR ? 2 : 1;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(static_cast<unsigned>(64 + 32 * a.epi_warps), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    attr[0] = pdl_attribute();
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(csize);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = PAIR ? 2 : 1;
    // as many units (CTAs, or pairs) as fit at once on the device, at most one per tile
    int units = sm_count() / csize;
    if (PAIR) {
        // how many pairs fit at once: one query per device, shared-memory size and block size
        static std::mutex mu;
        static int cached_smem[128] = {}, cached_fit[128] = {};
        const int key = smem * 16 + a.epi_warps;
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) dev = 0;
        int fit = 0;
        {
            std::lock_guard<std::mutex> lock(mu);
            if (cached_smem[dev] == key) {
                fit = cached_fit[dev];
            } else {
                cfg.gridDim = dim3(static_cast<unsigned>(units * csize), 1, 1);
                if (cudaOccupancyMaxActiveClusters(&fit, kern, &cfg) != cudaSuccess) fit = 0;
                cached_smem[dev] = key;
                cached_fit[dev] = fit;
            }
        }
        if (fit > 0 && fit < units) units = fit;
    }
    if (units > a.num_super) units = a.num_super;
    if (units < 1) units = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(units * csize), 1, 1);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, mp.a3, mp.b3, mp.a2, mp.b2, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int CODE, int LAYOUT, bool PAIR>
cudaError_t launch_out(const Maps &mp, const TcArgs &a, bt_dtype out_t, cudaStream_t s) {
    switch (out_t) {
        case BT_F32: return launch_t<CODE, LAYOUT, BT_F32, PAIR>(mp, a, s);
        case BT_BF16: return launch_t<CODE, LAYOUT, BT_BF16, PAIR>(mp, a, s);
        case BT_F16: return launch_t<CODE, LAYOUT, BT_F16, PAIR>(mp, a, s);
        default: return launch_t<CODE, LAYOUT, BT_I32, PAIR>(mp, a, s);
    }
}

template <int LAYOUT>
cudaError_t launch_code(bt_code code, bool pair, const Maps &mp, const TcArgs &a, bt_dtype out_t, cudaStream_t s) {
    if (code == BT_CODE_E4M3)
        return pair ? launch_out<BT_CODE_E4M3, LAYOUT, true>(mp, a, out_t, s)
                    : launch_out<BT_CODE_E4M3, LAYOUT, false>(mp, a, out_t, s);
    return pair ? launch_out<BT_CODE_E2M1, LAYOUT, true>(mp, a, out_t, s)
                : launch_out<BT_CODE_E2M1, LAYOUT, false>(mp, a, out_t, s);
}

int out_elem_bytes(bt_dtype t) { return t == BT_BF16 || t == BT_F16 ? 2 : 4; }

// Plan the tiles of an M x N contraction over rows of rb bytes (a multiple of
// 16; A and B rows pitch_a and pitch_b bytes apart) and encode the maps. With
// rb_split > 0 the contraction is split along K into parts of rb_split bytes
// (a multiple of 128) that the caller runs as K splits.
bool plan(TcArgs &a, Maps &mp, TileCfg &c, int code, const uint8_t *ap, const uint8_t *bp, int64_t M, int64_t N,
          int64_t rb, int64_t pitch_a, int64_t pitch_b, int out_elem, int64_t rb_split = -1,
          const TcTileChoice *pick = nullptr) {
    const int splits = rb_split > 0 ? static_cast<int>(rb / rb_split) : 1;
    if (rb % 16 != 0 || pitch_a % 16 != 0 || pitch_b % 16 != 0 || pitch_a < rb || pitch_b < rb ||
        M > (int64_t(1) << 31) - 512 || N > (int64_t(1) << 31) - 512)
        return false;
    a.M = M;
    a.N = N;
    if (rb_split > 0 && (rb_split % kRowB != 0 || rb % rb_split != 0)) return false;
    a.slices = static_cast<int>(((rb_split > 0 ? rb_split : rb) + kRowB - 1) / kRowB);   // per K split
    a.full_slices = static_cast<int>(rb / kRowB);                                       // of the whole row
    const int max_bn = code == BT_CODE_E2M1 ? 240 : 256;       // E2M1 keeps 32 TMEM columns for block scales
    c = choose_cfg(M, N, a.slices, sm_count(), max_bn, out_elem, splits, pick);
    // the shape's epilogue warp count when it is the one taken (0: the usual rule)
    a.epi_warps = (pick != nullptr && c.pair == (pick->pair != 0) && c.bn == pick->bn && c.d == pick->d) ? pick->epi : 0;
    a.bn = c.bn;
    a.d = c.d;
    a.nk = (a.slices + a.d - 1) / a.d;
    const int rows = c.pair ? 2 * kBM : kBM;
    const int64_t num_m = (M + rows - 1) / rows, num_n = (N + c.bn - 1) / c.bn;
    if (num_m * num_n > (int64_t(1) << 30)) return false;
    a.num_n = static_cast<int>(num_n);
    a.num_super = static_cast<int>(num_m * num_n);
    a.num_tiles = a.num_super;
    a.split_out = 0;
    a.idesc = make_idesc(code, rows, a.bn);
    const uint32_t b_box = static_cast<uint32_t>(b_slot_rows(a.bn, c.pair));
    return map_3d(&mp.a3, ap, static_cast<uint64_t>(pitch_a), static_cast<uint64_t>(M),
                  static_cast<uint64_t>(a.full_slices), kBM, static_cast<uint32_t>(a.d)) &&
           map_3d(&mp.b3, bp, static_cast<uint64_t>(pitch_b), static_cast<uint64_t>(N),
                  static_cast<uint64_t>(a.full_slices), b_box, static_cast<uint32_t>(a.d)) &&
           map_2d(&mp.a2, ap, static_cast<uint64_t>(rb), static_cast<uint64_t>(pitch_a), static_cast<uint64_t>(M), kBM) &&
           map_2d(&mp.b2, bp, static_cast<uint64_t>(rb), static_cast<uint64_t>(pitch_b), static_cast<uint64_t>(N), b_box);
}

// Measured shapes of the linear contraction (bt_tune_linear), keyed by the
// device and the problem, and the calling thread's forced shape.
struct TunedKey {
    int dev;
    int64_t M, N, K;
    int code, out_t;
    bool operator<(const TunedKey &o) const {
        if (dev != o.dev) return dev < o.dev;
        if (M != o.M) return M < o.M;
        if (N != o.N) return N < o.N;
        if (K != o.K) return K < o.K;
        if (code != o.code) return code < o.code;
        return out_t < o.out_t;
    }
};
std::mutex g_tuned_mu;
std::map<TunedKey, TcTileChoice> g_tuned;
std::atomic<int> g_tuned_count{0};          // entries: the common case (none) takes no lock
thread_local const TcTileChoice *t_forced = nullptr;

TunedKey tuned_key(int64_t M, int64_t N, int64_t K, bt_code code, bt_dtype out_t) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
    return TunedKey{dev, M, N, K, static_cast<int>(code), static_cast<int>(out_t)};
}

// The shape a linear contraction takes: the thread's forced one, else the
// measured winner for its key, else none (the cost model decides).
bool linear_pick(int64_t M, int64_t N, int64_t K, bt_code code, bt_dtype out_t, TcTileChoice &pick) {
    if (t_forced != nullptr) {
        pick = *t_forced;
        return true;
    }
    if (g_tuned_count.load(std::memory_order_acquire) == 0) return false;
    const TunedKey key = tuned_key(M, N, K, code, out_t);
    std::lock_guard<std::mutex> lock(g_tuned_mu);
    auto it = g_tuned.find(key);
    if (it == g_tuned.end()) return false;
    pick = it->second;
    return true;
}

}  // namespace

bool tc_available() { return encode_tiled() != nullptr; }

int tc_linear_candidates(int64_t M, int64_t N, int64_t K, bt_code code, bt_dtype out_t, TcTileChoice *out,
                         int max) {
    if (out == nullptr || max < 1 || M < 1 || N < 1 || K < 1 || (code != BT_CODE_E4M3 && code != BT_CODE_E2M1))
        return 0;
    const int max_bn = code == BT_CODE_E2M1 ? 240 : 256;
    const int oe = out_elem_bytes(out_t);
    const int slices = static_cast<int>((row_bytes(K, code) + kRowB - 1) / kRowB);
    const int sms = sm_count();
    // the model's own choice, with the epilogue warp count its launch takes
    const TileCfg first = choose_cfg(M, N, slices, sms, max_bn, oe, 1);
    TcArgs probe{};
    probe.slices = slices;
    probe.vec = (N * oe) % 16 == 0 ? 1 : 0;         // the output is 16-byte aligned
    const int epi0 = epilogue_warps(code, kRowsOut, probe);
    int n = 0;
    auto add = [&](bool pair, int bn, int d, int epi) {
        if (n >= max || !valid_shape(pair, bn, d, max_bn, oe, epi)) return;
        for (int i = 0; i < n; ++i)
            if (out[i].pair == (pair ? 1 : 0) && out[i].bn == bn && out[i].d == d && out[i].epi == epi) return;
        out[n++] = TcTileChoice{pair ? 1 : 0, bn, d, epi};
    };
    add(first.pair, first.bn, first.d, epi0);
    add(first.pair, first.bn, first.d, epi0 == 4 ? 8 : 4);
    for (int p = 1; p >= 0; --p)
        for (int d = 4; d >= 1; --d) {
            if ((p == 1) == first.pair && d == first.d) continue;
            int best_bn = 0;
            double best = -1.0;
            for (int bn = max_bn; bn >= 32; bn -= 16) {
                if (num_stages(bn, p == 1, d, oe) < 2) continue;
                const double cost = tile_cost(p == 1, bn, d, M, N, slices, sms, 1);
                if (best < 0.0 || cost < best * 0.999) {
                    best = cost;
                    best_bn = bn;
                }
            }
            if (best_bn == 0) continue;
            add(p == 1, best_bn, d, 4);
            add(p == 1, best_bn, d, 8);
        }
    // narrower tiles in the model's pairing and stage depth: more, shorter
    // tiles per SM, so less of the last tile's epilogue is left exposed
    for (int bn : {192, 160, 128, 112, 96})
        if (bn < first.bn) add(first.pair, bn, first.d, epi0);
    return n;
}

void tc_linear_force(const TcTileChoice *c) { t_forced = c; }

void tc_linear_remember(int64_t M, int64_t N, int64_t K, bt_code code, bt_dtype out_t, const TcTileChoice &c) {
    const TunedKey key = tuned_key(M, N, K, code, out_t);
    std::lock_guard<std::mutex> lock(g_tuned_mu);
    g_tuned[key] = c;
    g_tuned_count.store(static_cast<int>(g_tuned.size()), std::memory_order_release);
}

bool tc_linear_kept(int64_t M, int64_t N, int64_t K, bt_code code, bt_dtype out_t) {
    if (g_tuned_count.load(std::memory_order_acquire) == 0) return false;
    const TunedKey key = tuned_key(M, N, K, code, out_t);
    std::lock_guard<std::mutex> lock(g_tuned_mu);
    return g_tuned.find(key) != g_tuned.end();
}

void tc_linear_forget() {
    std::lock_guard<std::mutex> lock(g_tuned_mu);
    g_tuned.clear();
    g_tuned_count.store(0, std::memory_order_release);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() { return encode_tiled(); }

cudaError_t launch_tc_linear(const uint8_t *xp, const uint8_t *wp, bt_code code, int64_t M, int64_t N, int64_t K,
                             float alpha, void *out, bt_dtype out_t, unsigned int *err, cudaStream_t s,
                             const float *scales) {
    TcArgs a{};
    Maps mp;
    TileCfg c;
    const int64_t rb = row_bytes(K, code);
    TcTileChoice pick{};
    const bool picked = linear_pick(M, N, K, code, out_t, pick);
    if (!plan(a, mp, c, code, xp, wp, M, N, rb, rb, rb, out_elem_bytes(out_t), -1, picked ? &pick : nullptr))
        return cudaErrorInvalidValue;
    a.alpha = alpha;
    a.scales = scales;
    a.out = out;
    a.err = err;
    const int64_t ob = out_elem_bytes(out_t);
    a.vec = ((N * ob) % 16 == 0) && aligned(out, 16) ? 1 : 0;
    return launch_code<kRowsOut>(code, c.pair, mp, a, out_t, s);
}

cudaError_t launch_tc_conv(const uint8_t *rows, const uint8_t *wp, bt_code code, const ConvGeom &g, float alpha,
                           void *out, bt_dtype out_t, unsigned int *err, cudaStream_t s, const float *scales) {
    // D = W x rows^T: rows of the tile are output channels, columns output pixels.
    const int64_t krow = static_cast<int64_t>(g.k) * g.k * row_bytes(g.C, code);
    TcArgs a{};
    Maps mp;
    TileCfg c;
    if (!plan(a, mp, c, code, wp, rows, g.O, g.B * g.Ho * g.Wo, krow, krow, krow, out_elem_bytes(out_t)))
        return cudaErrorInvalidValue;
    a.alpha = alpha;
    a.scales = scales;
    a.out = out;
    a.err = err;
    a.hw = g.Ho * g.Wo;
    // widest store of a run of one channel's pixels that keeps every run inside
    // one image and naturally aligned
    const int eb = out_elem_bytes(out_t);
    a.vec = eb;
    for (int v = 16; v > eb; v /= 2) {
        if ((a.hw * eb) % v == 0 && aligned(out, static_cast<size_t>(v))) { a.vec = v; break; }
    }
    return launch_code<kNchwOut>(code, c.pair, mp, a, out_t, s);
}

// bf16 contractions: row-major output (bf16 or f32), or bf16 times the mask.
namespace {
template <int LAYOUT, int OUT>
cudaError_t launch_bf16_t(bool pair, const Maps &mp, const TcArgs &a, cudaStream_t s) {
    return pair ? launch_t<kCodeBF16, LAYOUT, OUT, true>(mp, a, s) : launch_t<kCodeBF16, LAYOUT, OUT, false>(mp, a, s);
}
}  // namespace

cudaError_t launch_tc_bf16(const uint16_t *a_ptr, int64_t lda, const uint16_t *b_ptr, int64_t ldb, int64_t M,
                           int64_t N, int64_t klen, float alpha, void *out, bt_dtype out_t, const TcMask *mask,
                           unsigned int *err, cudaStream_t s) {
    TcArgs a{};
    Maps mp;
    TileCfg c;
    if (!plan(a, mp, c, kCodeBF16, reinterpret_cast<const uint8_t *>(a_ptr), reinterpret_cast<const uint8_t *>(b_ptr),
              M, N, klen * 2, lda * 2, ldb * 2, mask != nullptr ? 2 : out_elem_bytes(out_t)))
        return cudaErrorInvalidValue;
    a.alpha = alpha;
    a.out = out;
    a.err = err;
    a.vec = ((N * out_elem_bytes(out_t)) % 16 == 0) && aligned(out, 16) ? 1 : 0;
    if (mask != nullptr) {
        if (out_t != BT_BF16 || !a.vec || N % 8 != 0 || !aligned(mask->x, 16)) return cudaErrorInvalidValue;
        a.aux = mask->x;
        a.aux_scale = mask->scale_a;
        a.aux_norm = mask->norm;
        a.aux_sum = mask->sum;
        return mask->x_t == BT_F32 ? launch_bf16_t<kRowsMaskF32, BT_BF16>(c.pair, mp, a, s)
                                   : launch_bf16_t<kRowsMaskBf16, BT_BF16>(c.pair, mp, a, s);
    }
    return out_t == BT_F32 ? launch_bf16_t<kRowsOut, BT_F32>(c.pair, mp, a, s)
                           : launch_bf16_t<kRowsOut, BT_BF16>(c.pair, mp, a, s);
}

// Split-K: out [splits, M, N] fp32 holds each K split's partial sums (alpha
// applied); klen a multiple of 64 * splits.
cudaError_t launch_tc_bf16_splitk(const uint16_t *a_ptr, int64_t lda, const uint16_t *b_ptr, int64_t ldb, int64_t M,
                                  int64_t N, int64_t klen, int splits, float alpha, float *out, unsigned int *err,
                                  cudaStream_t s, int64_t nchw_hw) {
    if (splits < 1 || klen % (64 * splits) != 0) return cudaErrorInvalidValue;
    TcArgs a{};
    Maps mp;
    TileCfg c;
    if (!plan(a, mp, c, kCodeBF16, reinterpret_cast<const uint8_t *>(a_ptr), reinterpret_cast<const uint8_t *>(b_ptr),
              M, N, klen * 2, lda * 2, ldb * 2, 4, klen * 2 / splits))
        return cudaErrorInvalidValue;
    if (static_cast<int64_t>(a.num_tiles) * splits > (int64_t(1) << 30)) return cudaErrorInvalidValue;
    a.num_super = a.num_tiles * splits;
    a.split_out = M * N;
    a.alpha = alpha;
    a.out = out;
    a.err = err;
    if (nchw_hw > 0) {
        // columns are pixels of images of nchw_hw pixels: each split's part NCHW
        a.hw = nchw_hw;
        a.vec = 4;
        for (int v = 16; v > 4; v /= 2) {
            if ((nchw_hw * 4) % v == 0 && aligned(out, static_cast<size_t>(v))) { a.vec = v; break; }
        }
        return launch_bf16_t<kNchwOut, BT_F32>(c.pair, mp, a, s);
    }
    a.vec = (N % 4 == 0) && aligned(out, 16) ? 1 : 0;
    return launch_bf16_t<kRowsOut, BT_F32>(c.pair, mp, a, s);
}

}  // namespace bt
