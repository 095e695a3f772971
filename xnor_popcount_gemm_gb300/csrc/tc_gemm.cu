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
// Persistent, warp-specialised: one CTA per SM walks output tiles of
// 128 x BN (BN a multiple of 16, chosen per problem so the tiles spread evenly
// over the SMs). The fp32 accumulator is double-buffered in TMEM (2 x 240
// columns plus 32 of unit block scales for E2M1, 2 x 256 for E4M3), so a
// tile's epilogue -- and its output stores -- overlap the next tile's MMAs.
//   warp 0 lane 0   TMA producer: a ring of smem stages, each one 128- or
//                   64-byte-wide K slice of A (128 rows) and B (BN rows),
//                   written with the matching swizzle; it runs ahead across
//                   tile boundaries.
//   warp 1 lane 0   MMA issuer: per 32 bytes of a stage, one tcgen05.mma
//                   (M=128, N=BN) into the tile's accumulator buffer;
//                   tcgen05.commit frees the stage, and, after a tile's last
//                   stage, hands the buffer to the epilogue.
//   warps 2..5      epilogue: each drains its 32 TMEM lanes (rows), the next
//                   32-column box in flight while the current
//                   one is scaled and cast. A linear output goes through a
//                   swizzled 32 x 32 smem box so that whole row segments leave in
//                   16-byte stores; a convolution's NCHW output is stored
//                   straight from registers (consecutive lanes, consecutive
//                   pixels). Once drained, the buffer goes back to the MMA
//                   warp.
// For a convolution, A is the matrix of im2col rows (one per output pixel,
// k*k packed input pixels long) and B the weights packed as [O, k, k, C], so
// the producer is the same as for a linear layer.
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "bt_device.cuh"
#include "bt_internal.h"
#include "tc_ptx.cuh"

namespace bt {
namespace {

constexpr int kBM = 128, kMaxBN = 256;           // tile rows (= MMA M), widest tile
constexpr int kThreads = 192;                    // producer, MMA, 4 epilogue warps
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol = 480;                 // 32 columns of unit block scales (E2M1)
constexpr uint32_t kUnitScales = 0x7F7F7F7Fu;    // UE8M0 127 = 2^0 in every byte
constexpr int kSmemMax = 232448;                 // 227 KB opt-in per CTA
constexpr int kBoxBytes = 32 * 128;              // one epilogue staging box: 32 rows x 128 B
constexpr int kStagingBytes = 4 * kBoxBytes;     // one box per epilogue warp
constexpr int kReserve = 1024 /*alignment*/ + 256 /*barriers*/;

struct TcArgs {
    int64_t M, N;
    int nk;                    // K steps per tile (smem stages to consume)
    int num_n, num_tiles, bn;  // tile grid; BN (multiple of 32, <= 256)
    int cm, cn;                // cluster shape: CTAs sharing B (along M) x sharing A (along N)
    int num_sn, num_super;     // super-tiles (cm x cn tiles, one per cluster at a time)
    uint32_t idesc;            // instruction descriptor for M=128, N=BN
    float alpha;
    void *out;
    unsigned int *err;
    int vec_store;             // linear: 1 when output rows are 16-byte aligned (16-byte stores)
                               // conv: bytes each lane stores at once (a run of pixels of one channel)
    int64_t hw;                // conv: output pixels per image (Ho * Wo)
    int stages;                // smem ring depth
};

// Shared memory: S stages of A (128 rows) and B (BN rows) K slices of ROWB
// bytes, the epilogue staging boxes, barriers. S is as many stages as fit (at
// most 8): narrow tiles get a deeper ring.
constexpr int kMaxStages = 8;
int num_stages(int rowb, int bn) {
    const int s = (kSmemMax - kReserve - kStagingBytes) / ((kBM + bn) * rowb);
    return s > kMaxStages ? kMaxStages : s;
}
int smem_bytes(int rowb, int bn) { return num_stages(rowb, bn) * (kBM + bn) * rowb + kStagingBytes + kReserve; }

// TMEM column of the second accumulator buffer; also the largest BN.
template <int CODE> __host__ __device__ constexpr uint32_t acc_stride() { return CODE == BT_CODE_E2M1 ? 240u : 256u; }

// Instruction descriptor: D = F32, K-major A and B, M = 128, N = bn.
uint32_t make_idesc(bt_code code, int bn) {
    const uint32_t mn = ((static_cast<uint32_t>(bn) >> 3) << 17) | ((static_cast<uint32_t>(kBM) >> 4) << 24);
    if (code == BT_CODE_E4M3) return (1u << 4) | (0u << 7) | (0u << 10) | mn;       // E4M3 x E4M3
    return (1u << 7) | (1u << 10) | (1u << 23) | mn;   // block-scaled E2M1 x E2M1, UE8M0 scales, ids 0
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

// One output value (conv epilogue) from its accumulator.
template <int OUT>
__device__ __forceinline__ typename OutT<OUT>::type from_acc(float acc, float alpha) {
    if constexpr (OUT == BT_F32) return __fmul_rn(acc, alpha);
    else if constexpr (OUT == BT_BF16) return __float2bfloat16_rn(__fmul_rn(acc, alpha));
    else if constexpr (OUT == BT_F16) return __float2half_rn(__fmul_rn(acc, alpha));
    else return __float2int_rn(acc);
}

// The bits of one output value (conv epilogue staging), in the low bits.
template <int OUT>
__device__ __forceinline__ uint32_t out_bits(float acc, float alpha) {
    if constexpr (OUT == BT_F32 || OUT == BT_I32) return FromAcc<OUT>::bits(acc, alpha);
    else if constexpr (OUT == BT_BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(acc, alpha)));
    else return __half_as_ushort(__float2half_rn(__fmul_rn(acc, alpha)));
}

// Position of 16-byte chunk q of staging-box row `row`: the 128-byte swizzle
// (q ^ row % 8) for 4-byte outputs (128-byte rows), the 64-byte swizzle
// (q ^ (row / 2) % 4) for 2-byte outputs (64-byte rows) -- the layouts TMA
// expects for CU_TENSOR_MAP_SWIZZLE_128B / _64B.
template <int ELEM>
__device__ __forceinline__ uint32_t box_chunk(int q, int row) {
    return ELEM == 4 ? static_cast<uint32_t>(q ^ (row & 7)) : static_cast<uint32_t>(q ^ ((row >> 1) & 3));
}

template <int CODE, int ROWB, bool CONV, int OUT>
__global__ void __launch_bounds__(kThreads, 1)
tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
          const TcArgs a) {
    const int S = a.stages;
    const int bn = a.bn;
    constexpr uint32_t kABytes = kBM * ROWB;
    const uint32_t kBBytes = static_cast<uint32_t>(bn * ROWB);
    constexpr int kMmaPerStage = ROWB / 32;        // K = 32 bytes per MMA
    using T = typename OutT<OUT>::type;
    constexpr int kElem = sizeof(T);
    constexpr int kBoxInner = 32 * kElem;          // bytes of one staging-box row: 32 output columns

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sA = base, sB = base + S * kABytes;
    const uint32_t sStage = sB + S * kBBytes;                        // epilogue staging boxes
    const uint32_t bars = sStage + kStagingBytes;                    // full[S], empty[S], tfull[2], tempty[2], drain
    uint8_t *gbars = smem_raw + (bars - raw);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(gbars + 8 * (2 * S + 5));
    volatile uint32_t *abort_flag = tmem_slot + 1;
    auto full = [&](int s) { return bars + 8u * s; };
    auto empty = [&](int s) { return bars + 8u * (S + s); };
    auto tfull = [&](int b) { return bars + 8u * (2 * S + b); };          // accumulator buffer b written
    auto tempty = [&](int b) { return bars + 8u * (2 * S + 2 + b); };     // accumulator buffer b drained
    const uint32_t drain = bars + 8u * (2 * S + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            tc::mbar_init(full(s), 1);
            // released by every CTA this one's copies land in (itself, its A
            // sharers and its B sharers)
            tc::mbar_init(empty(s), static_cast<uint32_t>(a.cm + a.cn - 1));
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(tfull(b), 1);
            tc::mbar_init(tempty(b), 4);   // one arrival per epilogue warp
        }
        tc::mbar_init(drain, 1);
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
    const bool clustered = a.cm * a.cn > 1;
    if (clustered) tc::cluster_sync();        // peers' barriers exist before any multicast lands
    const uint32_t tmem = *tmem_slot;
    // position in the cluster: rm along M (B sharers), rn along N (A sharers)
    const int crank = clustered ? static_cast<int>(tc::cluster_ctarank()) : 0;
    const int rm = crank % a.cm, rn = crank / a.cm;
    const int cluster = clustered ? static_cast<int>(tc::cluster_id_x()) : static_cast<int>(blockIdx.x);
    const int nclusters = clustered ? static_cast<int>(tc::num_clusters_x()) : static_cast<int>(gridDim.x);
    uint16_t maskA = 0, maskB = 0;
    for (int j = 0; j < a.cn; ++j) maskA |= static_cast<uint16_t>(1u << (rm + a.cm * j));
    for (int j = 0; j < a.cm; ++j) maskB |= static_cast<uint16_t>(1u << (j + a.cm * rn));
    const uint16_t mask_release = maskA | maskB;
    const int a_rows = kBM / a.cn;            // rows of the A tile this CTA loads
    const int b_rows = a.bn / a.cm;           // rows of the B tile this CTA loads
    const int quarter = warp & 3;                                   // TMEM lanes this warp may touch
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;

    if (CODE == BT_CODE_E2M1) {
        if (warp >= 2) {
            // unit block scales for A and B: every byte of columns [256, 288)
            tc::tmem_st16_fill(tmem + lane_base + kSfCol, kUnitScales);
            tc::tmem_st16_fill(tmem + lane_base + kSfCol + 16, kUnitScales);
            tc::tmem_st_wait();
        }
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
    }

    const uint32_t tx_bytes = static_cast<uint32_t>((kBM + bn) * ROWB);

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            pdl_wait();                                   // operands come from the previous kernel
            int s = 0;                                    // ring slot and its phase
            uint32_t ph = 0;
            uint32_t last_phase[kMaxStages];              // phase of each slot's last copy; 2 = none
#pragma unroll
            for (int i = 0; i < kMaxStages; ++i) last_phase[i] = 2u;
            bool ok = true;
            for (int st = cluster; st < a.num_super && ok; st += nclusters) {
                const int mt = (st / a.num_sn) * a.cm + rm, nt = (st % a.num_sn) * a.cn + rn;
                // this CTA's share of the A tile starts a_rows * rn rows in
                const int64_t am0 = static_cast<int64_t>(mt) * kBM + static_cast<int64_t>(a_rows) * rn;
                const int bn0 = nt * bn + b_rows * rm;                       // and of the B tile
                const uint32_t a_off = static_cast<uint32_t>(a_rows * rn * ROWB);
                const uint32_t b_off = static_cast<uint32_t>(b_rows * rm * ROWB);
                for (int kb = 0; kb < a.nk; ++kb) {
                    if (!tc::wait_bounded(empty(s), ph ^ 1u, abort_flag, a.err)) { ok = false; break; }
                    tc::mbar_arrive_expect_tx(full(s), tx_bytes);
                    const uint32_t adst = sA + s * kABytes + a_off, bdst = sB + s * kBBytes + b_off;
                    if (a.cn > 1) tc::tma_load_2d_mc(adst, &tmA, kb * ROWB, static_cast<int>(am0), full(s), maskA);
                    else tc::tma_load_2d(adst, &tmA, kb * ROWB, static_cast<int>(am0), full(s));
                    if (a.cm > 1) tc::tma_load_2d_mc(bdst, &tmB, kb * ROWB, bn0, full(s), maskB);
                    else tc::tma_load_2d(bdst, &tmB, kb * ROWB, bn0, full(s));
                    last_phase[s] = ph;
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                // let every issued copy land before the CTA can exit
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
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int s = 0;
            uint32_t ph = 0;
            int local = 0;
            bool ok = true;
            for (int st = cluster; st < a.num_super && ok; st += nclusters, ++local) {
                const int buf = local & 1;
                if (local >= 2) {
                    // the epilogue has drained this buffer (two tiles ago)
                    if (!tc::wait_bounded(tempty(buf), static_cast<uint32_t>((local - 2) >> 1) & 1u, abort_flag, a.err))
                        break;
                    tc::fence_after_sync();
                }
                const uint32_t dacc = tmem + static_cast<uint32_t>(buf) * acc_stride<CODE>();
                for (int kb = 0; kb < a.nk; ++kb) {
                    if (!tc::wait_bounded(full(s), ph, abort_flag, a.err)) { ok = false; break; }
                    tc::fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < kMmaPerStage; ++kk) {
                        const uint64_t bd = operand_desc<ROWB>(sB + s * kBBytes + kk * 32);
                        const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
                        const uint64_t ad = operand_desc<ROWB>(sA + s * kABytes + kk * 32);
                        if (CODE == BT_CODE_E4M3) tc::mma_f8f6f4(dacc, ad, bd, a.idesc, acc);
                        else tc::mma_mxf4(dacc, ad, bd, a.idesc, tmem + kSfCol, tmem + kSfCol + 16, acc);
                    }
                    if (clustered) tc::mma_commit_mc(empty(s), mask_release);
                    else tc::mma_commit(empty(s));
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
                if (ok) tc::mma_commit(tfull(buf));
            }
            // every MMA issued must finish before the accumulator is freed
            tc::mma_commit(drain);
            const unsigned long long t0 = globaltimer_ns();
            while (!tc::mbar_try_wait(drain, 0u) && globaltimer_ns() - t0 < kWaitNs) {}
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        pdl_wait();                                       // the previous kernel may still use `out`
        T *out = static_cast<T *>(a.out);
        const uint32_t my_stage = sStage + static_cast<uint32_t>((warp - 2) * kBoxBytes);   // one box per warp
        int local = 0;
        for (int st = cluster; st < a.num_super; st += nclusters, ++local) {
            const int mt = (st / a.num_sn) * a.cm + rm, nt = (st % a.num_sn) * a.cn + rn;
            const int64_t m0 = static_cast<int64_t>(mt) * kBM;
            const int n0 = nt * bn;
            const int buf = local & 1;
            if (!tc::wait_bounded(tfull(buf), static_cast<uint32_t>(local >> 1) & 1u, abort_flag, a.err)) break;
            tc::fence_after_sync();
            bool released = false;
            auto release = [&]() {
                // every TMEM read of this tile is complete: hand the accumulators back
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(tempty(buf));
                released = true;
            };
            // Boxes of 32 rows x 32 columns; the TMEM read of the next box is in
            // flight while the current one is converted and stored.
            const int64_t ncols = a.N - n0 < bn ? a.N - n0 : bn;
            const int64_t ncol_end = n0 + ncols;                             // this tile's columns end here
            const int nbox = ncols > 0 ? static_cast<int>((ncols + 31) / 32) : 0;
            const int64_t mrow0 = m0 + quarter * 32;                         // this warp's first row
            const int total = mrow0 < a.M ? nbox : 0;
            const uint32_t tbase = tmem + lane_base + static_cast<uint32_t>(buf) * acc_stride<CODE>();
            auto tcol_of = [&](int b) { return tbase + static_cast<uint32_t>(32 * b); };
            // conv: the output run this lane stores. With vw > kElem, a run of
            // vw / kElem pixels of one channel (vw bytes), starting at row
            // m = mrow0 + q * (vw / kElem) of the warp's 32; runs never straddle two
            // images (hw is a multiple of the run). Otherwise one pixel, m = mrow0 + lane.
            const int vw = CONV ? a.vec_store : 0;
            const bool runs = CONV && vw > kElem;
            const int lpr = runs ? kBoxInner / vw : 32;                      // lanes per staged channel row
            const int q = lane % lpr;
            const int64_t m = mrow0 + (runs ? q * (vw / kElem) : lane);
            const bool row_ok = m < a.M;
            T *pix_out = out;
            if constexpr (CONV) {
                const int64_t ob = row_ok ? m / a.hw : 0;
                pix_out = out + (ob * a.N + n0) * a.hw + (m - ob * a.hw);
            }
            auto emit = [&](const uint32_t (&r)[32], int b) {
                const int c0 = 32 * b;
                if constexpr (CONV) {
                    if (!runs) {
                        // NCHW: one store per channel, 32 consecutive pixels across the warp
                        if (!row_ok) return;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (c0 + j < ncols)
                                pix_out[static_cast<int64_t>(c0 + j) * a.hw] = from_acc<OUT>(__uint_as_float(r[j]), a.alpha);
                        return;
                    }
                    // NCHW through the staging box, transposed to [channel][pixel]
                    // rows; then each lane stores its run of one channel, 32 / lpr
                    // channels per instruction
                    const uint32_t sbox = my_stage;
                    __syncwarp();                                             // previous box fully read back
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const uint32_t addr = sbox + static_cast<uint32_t>(j * kBoxInner + lane * kElem);
                        const uint32_t v = out_bits<OUT>(__uint_as_float(r[j]), a.alpha);
                        if (kElem == 4) asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
                        else asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(static_cast<uint16_t>(v)) : "memory");
                    }
                    __syncwarp();
                    if (!row_ok) return;
                    const int rows_per = 32 / lpr;
                    for (int rr = lane / lpr; rr < 32; rr += rows_per) {
                        if (c0 + rr >= ncols) break;
                        const uint32_t addr = sbox + static_cast<uint32_t>(rr * kBoxInner + q * vw);
                        uint8_t *dst = reinterpret_cast<uint8_t *>(pix_out + static_cast<int64_t>(c0 + rr) * a.hw);
                        if (vw == 16) {
                            uint4 v;
                            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
                            *reinterpret_cast<uint4 *>(dst) = v;
                        } else if (vw == 8) {
                            uint2 v;
                            asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
                            *reinterpret_cast<uint2 *>(dst) = v;
                        } else {
                            uint32_t v;
                            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
                            *reinterpret_cast<uint32_t *>(dst) = v;
                        }
                    }
                } else {
                    // row-major [M, N] through the warp's swizzled staging box
                    const uint32_t sbox = my_stage;
                    __syncwarp();                                             // previous box fully read back
                    constexpr int kChunks = kBoxInner / 16;
#pragma unroll
                    for (int q = 0; q < kChunks; ++q) {
                        const uint32_t addr = sbox + static_cast<uint32_t>(lane * kBoxInner) + (box_chunk<kElem>(q, lane) << 4);
                        const uint4 w = chunk16<OUT, kElem>(r, q * (16 / kElem), a.alpha);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w.x), "r"(w.y),
                                     "r"(w.z), "r"(w.w)
                                     : "memory");
                    }
                    __syncwarp();
                    if (a.vec_store) {
                        // aligned rows: read the box back as 16-byte chunks, kChunks lanes
                        // per row, 32/kChunks rows per instruction, and store them whole
                        constexpr int kRowsPer = 32 / kChunks;
                        const int q = lane % kChunks;
                        const int64_t col = n0 + c0 + q * (16 / kElem);
#pragma unroll
                        for (int rr0 = 0; rr0 < 32; rr0 += kRowsPer) {
                            const int rr = rr0 + lane / kChunks;
                            const uint32_t addr = sbox + static_cast<uint32_t>(rr * kBoxInner) + (box_chunk<kElem>(q, rr) << 4);
                            uint4 v;
                            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                                         : "r"(addr));
                            const int64_t row = mrow0 + rr;
                            if (row < a.M && col < ncol_end)
                                st_stream_v4(reinterpret_cast<uint8_t *>(out) + (row * a.N + col) * kElem, v);
                        }
                    } else {
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
    }

    tc::fence_before_sync();
    __syncthreads();
    // no CTA leaves while a peer may still multicast into it or release its stages
    if (clustered) tc::cluster_sync();
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

int sm_count() {
    static int n[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
    if (n[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        n[dev] = v;
    }
    return n[dev];
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

// Tile configuration: BN (a multiple of 16 up to 240 for E2M1 / 256 for E4M3;
// the epilogue masks the part of its last 32-column box past the tile) and the
// cluster shape CM x CN. The cost
// model: a problem takes `rounds` waves of super-tiles over the clusters;
// each K stage costs the largest of its MMA time (one M=128 MMA per 32 bytes,
// about 116 clocks on GB300 whatever N up to 256), the time for the whole
// stage to land in this SM's shared memory (about 95 bytes per clock per SM
// for TMA into the ring; multicast inside a cluster lowers L2 reads but not
// the bytes each SM receives, so clusters only change the wave count), and
// the pipelined stage time measured in whole launches on GB300 (about 1230
// clocks per 128-byte stage and 790 per 64-byte stage, so 64-byte stages only
// pay off when they save a half-empty last stage of many); with the
// accumulator double-buffered only the last tile's epilogue (about 8 clocks
// per output column) is exposed.
// BT_TC_CONFIG="cm,cn,bn" overrides the choice.
struct TileCfg {
    int cm, cn, bn;
    double cost;     // modelled clocks of the whole launch
};

TileCfg choose_cfg(int64_t M, int64_t N, int nk, int rowb, int sms, int max_bn) {
    TileCfg best{1, 1, max_bn, 0.0};
    if (const char *env = std::getenv("BT_TC_CONFIG")) {
        int cm = 0, cn = 0, bn = 0;
        if (std::sscanf(env, "%d,%d,%d", &cm, &cn, &bn) == 3 && (cm == 1 || cm == 2) && (cn == 1 || cn == 2) &&
            bn >= 32 && bn <= max_bn && bn % 16 == 0 && (bn / cm) % 16 == 0)
            return TileCfg{cm, cn, bn, 0.0};
    }
    const int64_t num_m = (M + kBM - 1) / kBM;
    double best_cost = -1.0;
    for (int cm = 1; cm <= 2; ++cm) {
        for (int cn = 1; cn <= 2; ++cn) {
            const int64_t clusters = sms / (cm * cn);
            for (int bn = max_bn; bn >= 32; bn -= 16) {
                if ((bn / cm) % 16 != 0) continue;           // B slice rows: whole 16-row groups
                const int64_t num_n = (N + bn - 1) / bn;
                const int64_t super = ((num_m + cm - 1) / cm) * ((num_n + cn - 1) / cn);
                const int64_t rounds = (super + clusters - 1) / clusters;
                const double mma = (rowb / 32) * 116.0;
                const double land = static_cast<double>(kBM + bn) * rowb / 95.0;
                const double piped = 350.0 + 880.0 * rowb / 128.0;
                double stage = mma > land ? mma : land;
                if (piped > stage) stage = piped;
                const double cost = static_cast<double>(rounds) * nk * stage + 8.0 * bn + 600.0;
                if (best_cost < 0.0 || cost < best_cost * 0.999) {
                    best_cost = cost;
                    best = TileCfg{cm, cn, bn, cost};
                }
            }
        }
    }
    return best;
}

template <int CODE, int ROWB, bool CONV, int OUT>
cudaError_t launch_t(const CUtensorMap &ma, const CUtensorMap &mb, TcArgs a, cudaStream_t s) {
    auto kern = tc_kernel<CODE, ROWB, CONV, OUT>;
    a.stages = num_stages(ROWB, a.bn);
    const int smem = smem_bytes(ROWB, a.bn);
    if (a.stages < 2 || smem > kSmemMax) return cudaErrorInvalidValue;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] { attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax); });
    if (attr_err != cudaSuccess) return attr_err;
    const int csize = a.cm * a.cn;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(csize);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    // as many clusters as fit at once on the device, at most one per super-tile
    int clusters = sm_count() / csize;
    if (csize > 1) {
        cfg.gridDim = dim3(static_cast<unsigned>(clusters * csize), 1, 1);
        int fit = 0;
        if (cudaOccupancyMaxActiveClusters(&fit, kern, &cfg) == cudaSuccess && fit > 0 && fit < clusters) clusters = fit;
    }
    if (clusters > a.num_super) clusters = a.num_super;
    if (clusters < 1) clusters = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * csize), 1, 1);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int CODE, int ROWB, bool CONV>
cudaError_t launch_out(const CUtensorMap &ma, const CUtensorMap &mb, const TcArgs &a,
                       bt_dtype out_t, cudaStream_t s) {
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

int out_elem_bytes(bt_dtype t) { return t == BT_BF16 || t == BT_F16 ? 2 : 4; }

// Fill the tile-grid fields of `a` for configuration `c`.
bool set_grid(TcArgs &a, const TileCfg &c, int64_t M, int64_t N) {
    a.cm = c.cm;
    a.cn = c.cn;
    a.bn = c.bn;
    const int64_t num_m = (M + kBM - 1) / kBM, num_n = (N + c.bn - 1) / c.bn;
    const int64_t num_sn = (num_n + c.cn - 1) / c.cn;
    const int64_t num_super = ((num_m + c.cm - 1) / c.cm) * num_sn;
    if (num_super > (int64_t(1) << 30)) return false;
    a.num_n = static_cast<int>(num_n);
    a.num_tiles = static_cast<int>(num_m * num_n);
    a.num_sn = static_cast<int>(num_sn);
    a.num_super = static_cast<int>(num_super);
    return true;
}

}  // namespace

bool tc_available() { return encode_tiled() != nullptr; }

cudaError_t launch_tc_linear(const uint8_t *xp, const uint8_t *wp, bt_code code, int64_t M, int64_t N, int64_t K,
                             float alpha, void *out, bt_dtype out_t, unsigned int *err, cudaStream_t s) {
    const int64_t rb = row_bytes(K, code);
    TcArgs a{};
    a.M = M; a.N = N; a.nk = static_cast<int>((rb + 127) / 128); a.alpha = alpha; a.out = out; a.err = err;
    const int64_t ob = out_elem_bytes(out_t);
    a.vec_store = ((N * ob) % 16 == 0) && aligned(out, 16) ? 1 : 0;
    const TileCfg c = choose_cfg(M, N, a.nk, 128, sm_count(), code == BT_CODE_E2M1 ? 240 : 256);
    if (!set_grid(a, c, M, N)) return cudaErrorInvalidValue;
    a.idesc = make_idesc(code, a.bn);
    CUtensorMap ma, mb;
    if (!map_2d(&ma, xp, rb, rb, M, 128, static_cast<uint32_t>(kBM / a.cn)) ||
        !map_2d(&mb, wp, rb, rb, N, 128, static_cast<uint32_t>(a.bn / a.cm)))
        return cudaErrorInvalidValue;
    return launch_code<false>(code, 128, ma, mb, a, out_t, s);
}

cudaError_t launch_tc_conv(const uint8_t *rows, const uint8_t *wp, bt_code code, const ConvGeom &g, float alpha,
                           void *out, bt_dtype out_t, unsigned int *err, cudaStream_t s) {
    // A: the im2col rows [M, k*k*rbc]; B: the weights [O, k*k*rbc]. Rows are a
    // multiple of 64 bytes: 128-byte stages (the last one half zero fill when
    // the row is an odd number of 64-byte blocks) or 64-byte stages, whichever
    // the cost model prefers.
    const int64_t krow = static_cast<int64_t>(g.k) * g.k * row_bytes(g.C, code);
    if (krow % 64 != 0) return cudaErrorInvalidValue;
    TcArgs a{};
    a.M = g.B * g.Ho * g.Wo; a.N = g.O; a.alpha = alpha; a.out = out; a.err = err;
    a.hw = g.Ho * g.Wo;
    // widest store of a run of one channel's pixels that keeps every run inside
    // one image and naturally aligned
    const int eb = out_elem_bytes(out_t);
    a.vec_store = eb;
    for (int v = 16; v > eb; v /= 2) {
        if ((a.hw * eb) % v == 0 && aligned(out, static_cast<size_t>(v))) { a.vec_store = v; break; }
    }
    const int max_bn = code == BT_CODE_E2M1 ? 240 : 256;
    const int nk128 = static_cast<int>((krow + 127) / 128), nk64 = static_cast<int>(krow / 64);
    TileCfg c = choose_cfg(a.M, a.N, nk128, 128, sm_count(), max_bn);
    int rowb = 128;
    a.nk = nk128;
    if (krow % 128 != 0) {
        const TileCfg c64 = choose_cfg(a.M, a.N, nk64, 64, sm_count(), max_bn);
        if (c64.cost < c.cost) { c = c64; rowb = 64; a.nk = nk64; }
    }
    if (!set_grid(a, c, a.M, a.N)) return cudaErrorInvalidValue;
    a.idesc = make_idesc(code, a.bn);
    CUtensorMap ma, mb;
    if (!map_2d(&ma, rows, krow, krow, a.M, static_cast<uint32_t>(rowb), static_cast<uint32_t>(kBM / a.cn)) ||
        !map_2d(&mb, wp, krow, krow, g.O, static_cast<uint32_t>(rowb), static_cast<uint32_t>(a.bn / a.cm)))
        return cudaErrorInvalidValue;
    return launch_code<true>(code, rowb, ma, mb, a, out_t, s);
}

}  // namespace bt
