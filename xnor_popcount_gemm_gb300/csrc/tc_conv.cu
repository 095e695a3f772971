// Implicit-im2col binary convolution on the tensor cores (tcgen05), straight
// from channel-packed NHWC pixels: no im2col matrix is ever written.
//
// What it computes is the unfold + mm lowering of the im2col write-up
// (banghao.live/blog/9, section 2, MyConv2d.forward) on +1/-1 codes:
//   dot[b, o, i, j] = sum over taps (kh, kw) and channels c of
//                     w[o, kh, kw, c] * x[b, i*s - p + kh*d, j*s - p + kw*d, c]
// with taps that fall in the padding contributing 0, followed by the
// epilogue y = fp32(dot * alpha) cast to the output type (bitorch-engine
// BinaryConv2dForward.forward: the native result scaled by
// scale_a * scale_w, then .to(x.dtype)).
//
// The weights are the A operand (M = 128 output channels per tile, K-major
// rows [k, k, C] of E2M1 / E4M3 codes); the pixels are the B operand. A tile
// is 128 output channels x a band of `ht` output rows of one image. Its
// accumulator columns are "virtual pixels" v = i * wv + j of a row width wv >=
// Wo: the columns j >= Wo are computed and thrown away. In exchange every
// filter tap reads the same staged image, shifted by a whole number of rows:
//   stride s splits the input into s x s phase images (rows y = s*r + py,
//   columns x = s*u + px); tap (kh, kw) reads phase ((-p + kh*d) mod s,
//   (-p + kw*d) mod s) at phase coordinates (i + qy, j + qx) with
//   qy = floor((-p + kh*d) / s). Staging each phase image of the band as rows
//   of wv pixels starting at (qy_min, qx_min) makes the tap's B operand the
//   staged rows from (qy - qy_min) * wv + (qx - qx_min) on: one start
//   address, which the MMA descriptor takes as it is.
// Each phase image comes in with one TMA box per K slice: a 4-D tiled copy
// {slice bytes, wv columns, rv rows, 1 image} with traversal stride s along W
// and H, started at the band's (possibly negative) first coordinates, so the
// padding and the area past the image are zero-filled by the copy itself
// (code 0 = value 0: a padded tap adds nothing).
//
// Persistent, warp-specialised, one CTA per SM, single-CTA MMAs (M = 128):
//   warp 0 lane 0   TMA producer: the weights (resident for the whole launch
//                   when they fit beside two pixel stages, else a ring of
//                   slices re-read per tile) and a double-buffered stage of
//                   the tile's phase images;
//   warp 1 lane 0   MMA issuer: per tap and K slice, the MMAs of its 32-byte K
//                   steps into the tile's accumulator buffer (double-buffered
//                   in TMEM, so a tile's epilogue overlaps the next tile's MMAs);
//   warps 2..9      epilogue, two per TMEM lane quarter (32 channels) taking
//                   alternate 32-column boxes: scale and cast, stage the box in
//                   shared memory, read it back with lanes along the pixels and
//                   store each channel's valid pixels (consecutive addresses of
//                   one NCHW plane per store instruction).
// Every wait is bounded (bt_set_wait_timeout, 2 s by default; the teardown's
// drains of copies and MMAs in flight always 2 s): a wait that runs out
// records the timeout in the device error word and the kernel winds down
// without trapping.
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "bt_device.cuh"
#include "bt_internal.h"
#include "tc_ptx.cuh"

namespace bt {
namespace {

constexpr int kBM = 128;                          // output channels per tile (MMA M)
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol = 480;                  // E2M1: 32 columns of unit block scales
constexpr uint32_t kUnitScales = 0x7F7F7F7Fu;     // UE8M0 127 = 2^0 in every byte
constexpr int kSmemMax = 232448;                  // 227 KB opt-in per CTA
// One epilogue staging box per epilogue warp: 32 x 32 outputs (4 KB for
// 4-byte outputs, 2 KB for 2-byte ones).
__host__ __device__ constexpr int staging_bytes(int out_elem) { return kEpiWarps * 32 * 32 * out_elem; }
constexpr int kReserve = 1024 /*alignment*/ + 512 /*barriers*/;
constexpr int kMaxTaps = 64;
constexpr int kMaxPhases = 4;
constexpr int kMaxAStages = 8;
constexpr int kMaxBStages = 2;

struct ConvArgs {
    int B, O, Ho, Wo;
    int ht, bands;            // output rows per tile; tiles (bands) per image
    int wv;                   // virtual row width (>= Wo)
    int bn;                   // MMA N: accumulator columns per tile (multiple of 16, >= ht * wv)
    int num_ot, num_tiles;    // channel tiles (128 channels); tiles in all
    int ntap, nsl, sw;        // taps; K slices per tap; bytes per slice (64 or 128 = swizzle width)
    int nph;                  // phase images per tile
    int rv;                   // rows of virtual width staged per phase image
    int stride;               // convolution stride s (TMA traversal stride)
    uint32_t img_bytes;       // bytes of one (phase, slice) image, a multiple of 1024
    uint32_t stage_bytes;     // nph * nsl * img_bytes
    uint32_t img_tx;          // bytes one image's copy delivers: rv * wv * sw
    int b_stages;             // pixel stages (2, or 1 where two do not fit)
    int pairs;                // 2-byte outputs read back two pixels per lane (wv, Wo, Ho*Wo even)
    int a_resident;           // 1: every weight slice loaded once, kept for the launch
    int a_d;                  // slices per weight box
    int a_boxes;              // resident: boxes covering all slices
    int a_stages;             // streamed: ring depth
    int ph_x0[kMaxPhases];    // TMA start column of each phase image: s * qx_min + px
    int ph_y0[kMaxPhases];    // TMA start row relative to s * (first output row): s * qy_min + py
    uint32_t tap[kMaxTaps];   // (phase << 24) | first staged row the tap reads
    uint32_t idesc;
    float alpha;
    const float *scales;      // not null: alpha = fp32(scales[0] * scales[1])
    void *out;                // NCHW [B, O, Ho, Wo]
    unsigned int *err;
    unsigned long long wait_ns;  // limit of each bounded wait of the main loops (teardown drains: kWaitNs)
};

// Shared-memory matrix descriptor of a K-major operand in the 128- or 64-byte
// swizzle layout (rows of `sw` bytes, 8-row groups 8 * sw bytes apart). The
// start may sit on any row of a 1024-byte-aligned tile with the base-offset
// field left at 0: the swizzle is a function of the absolute shared-memory
// address bits, the same for the TMA copy that wrote the tile and for the MMA
// that reads it (checked on GB300 for row shifts 0..13 of both swizzles).
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t saddr, int sw) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(16u >> 4) << 16;                               // leading byte offset (unused)
    d |= static_cast<uint64_t>((8u * static_cast<uint32_t>(sw)) >> 4) << 32;  // stride byte offset
    d |= static_cast<uint64_t>(1u) << 46;                                     // descriptor version
    d |= static_cast<uint64_t>(sw == 128 ? 2u : 4u) << 61;                   // 128- / 64-byte swizzle
    return d;
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *m, int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// 16 bytes of converted outputs from accumulators r[j0 .. j0 + 16 / elem).
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

// Position of 16-byte chunk q of staging-box row `row` (rows of 32 outputs):
// swizzled so that 32 lanes writing their rows' chunk q hit distinct banks.
template <int ELEM>
__device__ __forceinline__ uint32_t box_chunk(int q, int row) {
    return ELEM == 4 ? static_cast<uint32_t>(q ^ (row & 7)) : static_cast<uint32_t>(q ^ ((row >> 1) & 3));
}

// Read back one staged box (32 channel rows x 32 virtual pixels) with lane =
// virtual pixel, and store row rr (channel o0 + rr) at p + rr * plane bytes,
// p being this lane's pixel in channel o0's output plane. All 32 shared loads
// go out before the stores; rows from nrows on (channels past O) and lanes
// whose pixel is not valid store nothing.
template <int ELEM>
__device__ __forceinline__ void box_to_planes(uint32_t sbox, int lane, bool valid, uint8_t *p, int64_t plane,
                                              int nrows) {
    constexpr int kBoxRow = 32 * ELEM;
    constexpr int kPer = 16 / ELEM;                      // outputs per 16-byte chunk
    const int q = lane / kPer;
    const uint32_t lane_off = sbox + static_cast<uint32_t>((lane % kPer) * ELEM);
    uint32_t v[32];
#pragma unroll
    for (int rr = 0; rr < 32; ++rr) {
        const uint32_t addr = lane_off + static_cast<uint32_t>(rr * kBoxRow) + (box_chunk<ELEM>(q, rr) << 4);
        if constexpr (ELEM == 4) {
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v[rr]) : "r"(addr));
        } else {
            uint16_t h;
            asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(addr));
            v[rr] = h;
        }
    }
    if (!valid) return;
    if (nrows >= 32) {
#pragma unroll
        for (int rr = 0; rr < 32; ++rr) {
            if constexpr (ELEM == 4) *reinterpret_cast<uint32_t *>(p) = v[rr];
            else *reinterpret_cast<uint16_t *>(p) = static_cast<uint16_t>(v[rr]);
            p += plane;
        }
    } else {
#pragma unroll
        for (int rr = 0; rr < 32; ++rr) {
            if (rr < nrows) {
                if constexpr (ELEM == 4) *reinterpret_cast<uint32_t *>(p) = v[rr];
                else *reinterpret_cast<uint16_t *>(p) = static_cast<uint16_t>(v[rr]);
            }
            p += plane;
        }
    }
}

// The same for 2-byte outputs, two virtual pixels per lane: lanes 0..15 take
// the 16 pixel pairs of even rows, lanes 16..31 of odd rows, so each shared
// load instruction reads two whole 64-byte rows and each store writes 4 bytes
// per lane. Needs wv, Wo and Ho * Wo even, so that a pair is either two valid
// pixels of one output row at an even offset or two dropped columns; p is
// this lane's pair in the plane of channel o0 + (lane >> 4).
__device__ __forceinline__ void box_to_planes_pairs(uint32_t sbox, int lane, bool valid, uint8_t *p, int64_t plane,
                                                    int nrows) {
    const int m = lane & 15, odd = lane >> 4;
    const uint32_t lane_off = sbox + static_cast<uint32_t>(odd * 64 + (m & 3) * 4);
    const int q = m >> 2;
    uint32_t v[16];
#pragma unroll
    for (int it = 0; it < 16; ++it) {
        const uint32_t addr = lane_off + static_cast<uint32_t>(it * 128) + (static_cast<uint32_t>(q ^ (it & 3)) << 4);
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v[it]) : "r"(addr));
    }
    if (!valid) return;
    const int64_t step = 2 * plane;
    if (nrows >= 32) {
#pragma unroll
        for (int it = 0; it < 16; ++it) {
            *reinterpret_cast<uint32_t *>(p) = v[it];
            p += step;
        }
    } else {
#pragma unroll
        for (int it = 0; it < 16; ++it) {
            if (2 * it + odd < nrows) *reinterpret_cast<uint32_t *>(p) = v[it];
            p += step;
        }
    }
}

template <int CODE, int OUT, int SW, bool PAIRS>
__global__ void __launch_bounds__(kThreads, 1)
conv_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const ConvArgs a) {
    using T = typename OutT<OUT>::type;
    constexpr int kElem = sizeof(T);
    constexpr int kBoxRow = 32 * kElem;              // bytes of one staging-box row
    constexpr uint32_t kASlice = kBM * SW;           // weight bytes per K slice
    constexpr int kMmaPerSlice = SW / 32;            // 32 bytes of K per MMA
    constexpr uint32_t kAccStride = CODE == BT_CODE_E2M1 ? 240u : 256u;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int nslices = a.ntap * a.nsl;
    const uint32_t a_bytes = a.a_resident ? static_cast<uint32_t>(a.a_boxes * a.a_d) * kASlice
                                          : static_cast<uint32_t>(a.a_stages * a.a_d) * kASlice;
    const uint32_t sA = base;
    const uint32_t sB = sA + a_bytes;
    const uint32_t sStage = sB + static_cast<uint32_t>(a.b_stages) * a.stage_bytes;
    const uint32_t bars = sStage + staging_bytes(kElem);
    // barriers: afull[8], aempty[8], bfull[2], bempty[2], tfull[2], tempty[2], drain
    auto afull = [&](int i) { return bars + 8u * i; };
    auto aempty = [&](int i) { return bars + 8u * (kMaxAStages + i); };
    auto bfull = [&](int i) { return bars + 8u * (2 * kMaxAStages + i); };
    auto bempty = [&](int i) { return bars + 8u * (2 * kMaxAStages + 2 + i); };
    auto tfull = [&](int i) { return bars + 8u * (2 * kMaxAStages + 4 + i); };
    auto tempty = [&](int i) { return bars + 8u * (2 * kMaxAStages + 6 + i); };
    const uint32_t drain = bars + 8u * (2 * kMaxAStages + 8);
    volatile uint32_t *tmem_slot =
        reinterpret_cast<volatile uint32_t *>(smem_raw + (bars - raw) + 8 * (2 * kMaxAStages + 9));
    volatile uint32_t *abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < kMaxAStages; ++i) {
            tc::mbar_init(afull(i), 1);
            tc::mbar_init(aempty(i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bfull(i), 1);
            tc::mbar_init(bempty(i), 1);
            tc::mbar_init(tfull(i), 1);
            tc::mbar_init(tempty(i), static_cast<uint32_t>(kEpiWarps));
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
    const uint32_t tmem = *tmem_slot;
    const int quarter = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    if (CODE == BT_CODE_E2M1 && warp >= 2 && warp < 6) {
        tc::tmem_st16_fill(tmem + lane_base + kSfCol, kUnitScales);
        tc::tmem_st16_fill(tmem + lane_base + kSfCol + 16, kUnitScales);
        tc::tmem_st_wait();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    const int unit = static_cast<int>(blockIdx.x), nunits = static_cast<int>(gridDim.x);
    const int hw = a.Ho * a.Wo;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            pdl_wait();                                   // pixels (and weights) come from earlier kernels
            int as = 0, bs = 0;
            uint32_t aph = 0, bph = 0;
            uint32_t a_last[kMaxAStages], b_last[2];      // phase of each slot's last copy; 2 = none
            for (int i = 0; i < kMaxAStages; ++i) a_last[i] = 2u;
            b_last[0] = b_last[1] = 2u;
            bool ok = true, a_loaded = false;
            for (int t = unit; t < a.num_tiles && ok; t += nunits) {
                const int ot = t % a.num_ot, rest = t / a.num_ot;
                const int b = rest / a.bands, band = rest - b * a.bands;
                const int r0 = band * a.ht;
                // the tile's phase images
                if (!tc::wait_bounded(bempty(bs), bph ^ 1u, abort_flag, a.err, a.wait_ns)) { ok = false; break; }
                tc::mbar_arrive_expect_tx(bfull(bs), static_cast<uint32_t>(a.nph * a.nsl) * a.img_tx);
                const uint32_t dst0 = sB + static_cast<uint32_t>(bs) * a.stage_bytes;
                for (int ph = 0; ph < a.nph; ++ph)
                    for (int sl = 0; sl < a.nsl; ++sl)
                        tma_load_4d(dst0 + static_cast<uint32_t>(ph * a.nsl + sl) * a.img_bytes, &tmB, sl * SW,
                                    a.ph_x0[ph], a.stride * r0 + a.ph_y0[ph], b, bfull(bs));
                b_last[bs] = bph;
                if (++bs == a.b_stages) { bs = 0; bph ^= 1u; }
                // resident weights: after the first tile's pixels, one barrier per
                // box (up to kMaxAStages boxes; more share the first barrier), so
                // that the first MMAs start once their taps have landed
                if (a.a_resident && !a_loaded) {
                    const bool per_box = a.a_boxes <= kMaxAStages;
                    if (!per_box)
                        tc::mbar_arrive_expect_tx(afull(0), static_cast<uint32_t>(a.a_boxes * a.a_d) * kASlice);
                    for (int i = 0; i < a.a_boxes; ++i) {
                        if (per_box) {
                            tc::mbar_arrive_expect_tx(afull(i), static_cast<uint32_t>(a.a_d) * kASlice);
                            a_last[i] = 0u;
                        }
                        tc::tma_load_3d(sA + static_cast<uint32_t>(i * a.a_d) * kASlice, &tmA, 0, ot * kBM,
                                        i * a.a_d, afull(per_box ? i : 0));
                    }
                    if (!per_box) a_last[0] = 0u;
                    a_loaded = true;
                }
                if (!a.a_resident) {
                    for (int i0 = 0; i0 < nslices; i0 += a.a_d) {
                        if (!tc::wait_bounded(aempty(as), aph ^ 1u, abort_flag, a.err, a.wait_ns)) { ok = false; break; }
                        tc::mbar_arrive_expect_tx(afull(as), static_cast<uint32_t>(a.a_d) * kASlice);
                        tc::tma_load_3d(sA + static_cast<uint32_t>(as * a.a_d) * kASlice, &tmA, 0, ot * kBM, i0,
                                        afull(as));
                        a_last[as] = aph;
                        if (++as == a.a_stages) { as = 0; aph ^= 1u; }
                    }
                }
            }
            if (!ok) {
                // let every issued copy land before the CTA can exit
                const unsigned long long t0 = globaltimer_ns();
                for (int i = 0; i < kMaxAStages; ++i)
                    if (a_last[i] < 2u)
                        while (!tc::mbar_try_wait(afull(i), a_last[i]) && globaltimer_ns() - t0 < kWaitNs) {}
                for (int i = 0; i < 2; ++i)
                    if (b_last[i] < 2u)
                        while (!tc::mbar_try_wait(bfull(i), b_last[i]) && globaltimer_ns() - t0 < kWaitNs) {}
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int as = 0, bs = 0, local = 0;
            uint32_t aph = 0, bph = 0;
            bool ok = true;
            for (int t = unit; t < a.num_tiles && ok; t += nunits, ++local) {
                const int buf = local & 1;
                if (local >= 2) {
                    if (!tc::wait_bounded(tempty(buf), static_cast<uint32_t>((local - 2) >> 1) & 1u, abort_flag, a.err, a.wait_ns))
                        break;
                    tc::fence_after_sync();
                }
                if (!tc::wait_bounded(bfull(bs), bph, abort_flag, a.err, a.wait_ns)) break;
                tc::fence_after_sync();
                const uint32_t dacc = tmem + static_cast<uint32_t>(buf) * kAccStride;
                // descriptors are built once and moved by adding (byte offset >> 4)
                // to their start-address field (shared-memory addresses stay below
                // 256 KB, so the 14-bit field never carries): the issuing thread
                // spends a few integer adds per MMA, not a descriptor build
                const uint64_t bdesc_stage = kmajor_desc(sB + static_cast<uint32_t>(bs) * a.stage_bytes, SW);
                const uint64_t adesc_base = kmajor_desc(sA, SW);
                const uint32_t img16 = a.img_bytes >> 4;
                constexpr uint32_t kSlice16 = kASlice >> 4;
                uint64_t adesc = adesc_base;
                int idx = 0, within = 0, box = 0;
                for (int tp = 0; tp < a.ntap && ok; ++tp) {
                    const uint32_t tapw = a.tap[tp];
                    uint64_t bd = bdesc_stage + (tapw >> 24) * static_cast<uint32_t>(a.nsl) * img16 +
                                  (tapw & 0xFFFFFFu) * (SW >> 4);
                    for (int sl = 0; sl < a.nsl; ++sl, ++idx) {
                        if (within == 0) {
                            if (a.a_resident) {
                                // first tile: each box of weights on its own barrier (or all on the first)
                                if (local == 0 && (a.a_boxes <= kMaxAStages || idx == 0)) {
                                    if (!tc::wait_bounded(afull(a.a_boxes <= kMaxAStages ? box : 0), 0u, abort_flag, a.err,
                                                          a.wait_ns)) { ok = false; break; }
                                    tc::fence_after_sync();
                                }
                                adesc = adesc_base + static_cast<uint64_t>(idx) * kSlice16;
                            } else {
                                if (!tc::wait_bounded(afull(as), aph, abort_flag, a.err, a.wait_ns)) { ok = false; break; }
                                tc::fence_after_sync();
                                adesc = adesc_base + static_cast<uint64_t>(as * a.a_d) * kSlice16;
                            }
                        }
#pragma unroll
                        for (int kk = 0; kk < kMmaPerSlice; ++kk) {
                            const uint32_t acc = (idx | kk) != 0 ? 1u : 0u;
                            if (CODE == BT_CODE_E4M3) tc::mma_f8f6f4(dacc, adesc + 2 * kk, bd + 2 * kk, a.idesc, acc);
                            else tc::mma_mxf4(dacc, adesc + 2 * kk, bd + 2 * kk, a.idesc, tmem + kSfCol, tmem + kSfCol + 16, acc);
                        }
                        adesc += kSlice16;
                        bd += img16;
                        if (++within == a.a_d) {
                            within = 0;
                            ++box;
                            if (!a.a_resident) {
                                tc::mma_commit(aempty(as));
                                if (++as == a.a_stages) { as = 0; aph ^= 1u; }
                            }
                        }
                    }
                }
                if (!ok) break;
                tc::mma_commit(bempty(bs));
                if (++bs == a.b_stages) { bs = 0; bph ^= 1u; }
                tc::mma_commit(tfull(buf));
            }
            // every MMA issued must finish before the accumulator is freed
            tc::mma_commit(drain);
            const unsigned long long t0 = globaltimer_ns();
            while (!tc::mbar_try_wait(drain, 0u) && globaltimer_ns() - t0 < kWaitNs) {}
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (warps 2..9) ----------------
        pdl_wait();                                       // the previous kernel may still use `out`
        T *const out = static_cast<T *>(a.out);
        const uint32_t sbox = sStage + static_cast<uint32_t>((warp - 2) * 32 * 32 * kElem);
        const float alpha = a.scales != nullptr ? alpha_from(a.scales) : a.alpha;
        const int half = (warp - 2) / 4;
        int local = 0;
        for (int t = unit; t < a.num_tiles; t += nunits, ++local) {
            const int ot = t % a.num_ot, rest = t / a.num_ot;
            const int b = rest / a.bands, band = rest - b * a.bands;
            const int r0 = band * a.ht;
            const int hte = a.Ho - r0 < a.ht ? a.Ho - r0 : a.ht;       // output rows of this band
            const int buf = local & 1;
            if (!tc::wait_bounded(tfull(buf), static_cast<uint32_t>(local >> 1) & 1u, abort_flag, a.err, a.wait_ns)) break;
            tc::fence_after_sync();
            const int o0 = ot * kBM + quarter * 32;                     // this warp's first channel
            const int nrows = a.O - o0 < 32 ? a.O - o0 : 32;
            const int ncols = hte * a.wv;
            const int nbox = (ncols + 31) / 32;
            const uint32_t tbase = tmem + lane_base + static_cast<uint32_t>(buf) * kAccStride;
            T *const plane0 = out + (static_cast<int64_t>(b) * a.O + o0) * hw + static_cast<int64_t>(r0) * a.Wo;
            if (nrows > 0) {
                for (int bx = half; bx < nbox; bx += 2) {
                    uint32_t r[32];
                    tc::tmem_ld32(tbase + static_cast<uint32_t>(32 * bx), r);
                    tc::tmem_ld_wait();
                    // stage: row = this lane's channel, 32 virtual pixels, swizzled
                    __syncwarp();
#pragma unroll
                    for (int q = 0; q < kBoxRow / 16; ++q) {
                        const uint32_t addr = sbox + static_cast<uint32_t>(lane * kBoxRow) + (box_chunk<kElem>(q, lane) << 4);
                        const uint4 w = chunk16<OUT, kElem>(r, q * (16 / kElem), alpha);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w.x), "r"(w.y),
                                     "r"(w.z), "r"(w.w)
                                     : "memory");
                    }
                    __syncwarp();
                    // read back with lanes along the pixels
                    if constexpr (PAIRS) {
                        const int v = 32 * bx + 2 * (lane & 15);
                        const int i = v / a.wv, j = v - i * a.wv;
                        const bool valid = v < ncols && j < a.Wo;
                        uint8_t *p = reinterpret_cast<uint8_t *>(plane0 + static_cast<int64_t>(lane >> 4) * hw +
                                                                 static_cast<int64_t>(i) * a.Wo + j);
                        box_to_planes_pairs(sbox, lane, valid, p, static_cast<int64_t>(hw) * kElem, nrows);
                    } else {
                        const int v = 32 * bx + lane;          // lane = virtual pixel
                        const int i = v / a.wv, j = v - i * a.wv;
                        const bool valid = v < ncols && j < a.Wo;
                        uint8_t *p = reinterpret_cast<uint8_t *>(plane0 + static_cast<int64_t>(i) * a.Wo + j);
                        box_to_planes<kElem>(sbox, lane, valid, p, static_cast<int64_t>(hw) * kElem, nrows);
                    }
                }
            }
            // every TMEM read of this tile is complete: hand the accumulator back
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tempty(buf));
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

uint32_t make_idesc(int code, int m, int bn) {
    const uint32_t mn = ((static_cast<uint32_t>(bn) >> 3) << 17) | ((static_cast<uint32_t>(m) >> 4) << 24);
    if (code == BT_CODE_E4M3) return (1u << 4) | mn;                             // E4M3 x E4M3 -> F32
    return (1u << 7) | (1u << 10) | (1u << 23) | mn;   // block-scaled E2M1 x E2M1, UE8M0 scales, ids 0
}

int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

struct ConvPlan {
    ConvArgs a;
    int smem;
    int grid;
};

// The implicit plan of a convolution, or false where it does not apply (the
// caller then unfolds explicitly): E2M1 / E4M3 codes, stride 1 or 2, at most
// 64 taps, a virtual row that fits one tile, copies within TMA's box limits,
// and shared memory for the weights (resident or a ring of at least two
// stages) beside two pixel stages and the epilogue's staging.
bool plan_conv(const ConvGeom &g, bt_code code, int sms, int out_elem, ConvPlan &p) {
    if (code != BT_CODE_E2M1 && code != BT_CODE_E4M3) return false;
    if (g.s < 1 || g.s > 2 || g.k < 1 || g.k * g.k > kMaxTaps) return false;
    if (g.B < 1 || g.B > (int64_t(1) << 24) || g.O < 1 || g.O > (int64_t(1) << 24)) return false;
    if (g.Ho < 1 || g.Wo < 1 || g.Ho > 65536 || g.Wo > 256 || g.H > (int64_t(1) << 30) || g.W > (int64_t(1) << 30))
        return false;
    const int64_t cb = row_bytes(g.C, code);
    const int sw = cb % 128 == 0 ? 128 : 64;
    if (cb % sw != 0) return false;
    ConvArgs &a = p.a;
    std::memset(&a, 0, sizeof(a));
    a.B = static_cast<int>(g.B);
    a.O = static_cast<int>(g.O);
    a.Ho = static_cast<int>(g.Ho);
    a.Wo = static_cast<int>(g.Wo);
    a.sw = sw;
    a.nsl = static_cast<int>(cb / sw);
    a.ntap = g.k * g.k;
    a.stride = g.s;
    if (static_cast<int64_t>(a.ntap) * a.nsl > 65535) return false;
    // phases and tap offsets (along one axis: e = -p + kk*d = s*q + ph)
    const int s = g.s;
    int phase_id[4] = {-1, -1, -1, -1};
    int qy_min[4], qx_min[4], qx_span = 0;
    int nph = 0;
    for (int kh = 0; kh < g.k; ++kh)
        for (int kw = 0; kw < g.k; ++kw) {
            const int ey = -g.p + kh * g.d, ex = -g.p + kw * g.d;
            const int qy = floor_div(ey, s), qx = floor_div(ex, s);
            const int key = (ey - s * qy) * 2 + (ex - s * qx);
            if (phase_id[key] < 0) {
                phase_id[key] = nph;
                qy_min[nph] = qy;
                qx_min[nph] = qx;
                a.ph_y0[nph] = s * qy + (ey - s * qy);
                a.ph_x0[nph] = s * qx + (ex - s * qx);
                ++nph;
            }
            const int id = phase_id[key];
            if (qy < qy_min[id]) { qy_min[id] = qy; a.ph_y0[id] = s * qy + (ey - s * qy); }
            if (qx < qx_min[id]) { qx_min[id] = qx; a.ph_x0[id] = s * qx + (ex - s * qx); }
        }
    a.nph = nph;
    int qy_off_max = 0, qx_off_max = 0;
    for (int kh = 0; kh < g.k; ++kh)
        for (int kw = 0; kw < g.k; ++kw) {
            const int ey = -g.p + kh * g.d, ex = -g.p + kw * g.d;
            const int qy = floor_div(ey, s), qx = floor_div(ex, s);
            const int id = phase_id[(ey - s * qy) * 2 + (ex - s * qx)];
            if (qy - qy_min[id] > qy_off_max) qy_off_max = qy - qy_min[id];
            if (qx - qx_min[id] > qx_off_max) qx_off_max = qx - qx_min[id];
        }
    qx_span = qx_off_max;
    a.wv = a.Wo + qx_span;
    const int bn_max = code == BT_CODE_E2M1 ? 240 : 256;
    // an even row width keeps pixel pairs of an even Wo aligned in the output
    if (a.Wo % 2 == 0 && a.wv % 2 == 1 && a.wv + 1 <= bn_max) a.wv += 1;
    if (a.wv > bn_max || a.wv * s > 256) return false;
    int ht = bn_max / a.wv;
    if (ht > a.Ho) ht = a.Ho;
    a.bands = (a.Ho + ht - 1) / ht;
    a.ht = (a.Ho + a.bands - 1) / a.bands;           // balance the bands
    a.bn = (a.ht * a.wv + 15) / 16 * 16;
    if (a.bn < 32) a.bn = 32;
    if (a.bn > bn_max) return false;
    int max_off = 0;
    for (int kh = 0; kh < g.k; ++kh)
        for (int kw = 0; kw < g.k; ++kw) {
            const int ey = -g.p + kh * g.d, ex = -g.p + kw * g.d;
            const int qy = floor_div(ey, s), qx = floor_div(ex, s);
            const int id = phase_id[(ey - s * qy) * 2 + (ex - s * qx)];
            const int off = (qy - qy_min[id]) * a.wv + (qx - qx_min[id]);
            a.tap[kh * g.k + kw] = (static_cast<uint32_t>(id) << 24) | static_cast<uint32_t>(off);
            if (off > max_off) max_off = off;
        }
    a.rv = (a.bn + max_off + a.wv - 1) / a.wv;
    if (a.rv * s > 256) return false;
    a.img_tx = static_cast<uint32_t>(a.rv * a.wv * sw);
    a.img_bytes = (a.img_tx + 1023u) / 1024u * 1024u;
    a.stage_bytes = static_cast<uint32_t>(a.nph * a.nsl) * a.img_bytes;
    a.num_ot = (a.O + kBM - 1) / kBM;
    const int64_t tiles = static_cast<int64_t>(a.num_ot) * a.B * a.bands;
    if (tiles > (int64_t(1) << 30)) return false;
    a.num_tiles = static_cast<int>(tiles);
    // weights resident (loaded once per CTA, each CTA keeping one channel
    // tile) or streamed through a ring of slices re-read per tile; one or two
    // pixel stages. Preference: resident + two stages; resident + one stage
    // when a CTA gets at most two tiles (only the second tile's copy is then
    // exposed); streamed + two stages; resident + one; streamed + one.
    // BT_CONV_PLAN=r2|r1|s2|s1 picks one where it fits.
    const int nslices = a.ntap * a.nsl;
    const int64_t slice_a = static_cast<int64_t>(kBM) * sw;
    int units = sms;
    if (units > a.num_tiles) units = a.num_tiles;
    int a_d_res = 1;
    for (int d = 8; d >= 1; --d)
        if (nslices % d == 0) { a_d_res = d; break; }
    const int64_t a_res_bytes = static_cast<int64_t>(nslices) * slice_a;
    auto fixed_of = [&](int bst) {
        return kReserve + staging_bytes(out_elem) + static_cast<int64_t>(bst) * a.stage_bytes;
    };
    auto fits_res = [&](int bst) { return units >= a.num_ot && fixed_of(bst) + a_res_bytes <= kSmemMax; };
    auto stream_d = [&](int bst, int *stages) {
        for (int d = 4; d >= 1; --d) {
            if (nslices % d != 0) continue;
            const int64_t room = kSmemMax - fixed_of(bst);
            const int64_t st = room > 0 ? room / (d * slice_a) : 0;
            if (st >= 2) { *stages = static_cast<int>(st > kMaxAStages ? kMaxAStages : st); return d; }
        }
        return 0;
    };
    int st2 = 0, st1 = 0;
    const int sd2 = stream_d(2, &st2), sd1 = stream_d(1, &st1);
    const bool few = a.num_tiles <= 2 * ((units / a.num_ot) * a.num_ot > 0 ? (units / a.num_ot) * a.num_ot : units);
    char plan = 0;                                   // 'R' resident, 'S' streamed
    int bst = 2;
    if (const char *env = std::getenv("BT_CONV_PLAN")) {
        if (std::strcmp(env, "r2") == 0 && fits_res(2)) { plan = 'R'; bst = 2; }
        else if (std::strcmp(env, "r1") == 0 && fits_res(1)) { plan = 'R'; bst = 1; }
        else if (std::strcmp(env, "s2") == 0 && sd2) { plan = 'S'; bst = 2; }
        else if (std::strcmp(env, "s1") == 0 && sd1) { plan = 'S'; bst = 1; }
    }
    if (plan == 0) {
        if (fits_res(2)) { plan = 'R'; bst = 2; }
        else if (few && fits_res(1)) { plan = 'R'; bst = 1; }
        else if (sd2) { plan = 'S'; bst = 2; }
        else if (fits_res(1)) { plan = 'R'; bst = 1; }
        else if (sd1) { plan = 'S'; bst = 1; }
        else return false;
    }
    a.b_stages = bst;
    if (plan == 'R') {
        a.a_resident = 1;
        a.a_d = a_d_res;
        a.a_boxes = nslices / a_d_res;
        a.a_stages = 0;
        units = units / a.num_ot * a.num_ot;
        p.smem = static_cast<int>(fixed_of(bst) + a_res_bytes);
    } else {
        a.a_resident = 0;
        a.a_boxes = 0;
        a.a_d = bst == 2 ? sd2 : sd1;
        a.a_stages = bst == 2 ? st2 : st1;
        p.smem = static_cast<int>(fixed_of(bst) + static_cast<int64_t>(a.a_stages) * a.a_d * slice_a);
    }
    if (p.smem > kSmemMax) return false;
    p.grid = units < 1 ? 1 : units;
    a.idesc = make_idesc(code, kBM, a.bn);
    a.pairs = (a.wv % 2 == 0 && a.Wo % 2 == 0 && (static_cast<int64_t>(a.Ho) * a.Wo) % 2 == 0) ? 1 : 0;
    return true;
}

bool encode_maps(const ConvGeom &g, bt_code code, const ConvArgs &a, const uint8_t *xp, const uint8_t *wp,
                 CUtensorMap *ma, CUtensorMap *mb) {
    auto fn = tensor_map_encoder();
    if (fn == nullptr) return false;
    const uint64_t cb = static_cast<uint64_t>(row_bytes(g.C, code));
    const CUtensorMapSwizzle swz = a.sw == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    // weights [O, k*k*cb] as {sw bytes, O rows, k*k*nsl slices}
    {
        cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.sw), static_cast<cuuint64_t>(g.O),
                              static_cast<cuuint64_t>(a.ntap * a.nsl)};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.ntap) * cb, static_cast<cuuint64_t>(a.sw)};
        cuuint32_t box[3] = {static_cast<cuuint32_t>(a.sw), static_cast<cuuint32_t>(kBM),
                             static_cast<cuuint32_t>(a.a_d)};
        cuuint32_t es[3] = {1, 1, 1};
        if (fn(ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(wp), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    // packed pixels [B, H, W, cb] as {cb bytes, W, H, B}; a box takes one slice
    // of wv columns and rv rows with traversal stride s
    {
        cuuint64_t dims[4] = {cb, static_cast<cuuint64_t>(g.W), static_cast<cuuint64_t>(g.H),
                              static_cast<cuuint64_t>(g.B)};
        cuuint64_t strides[3] = {cb, static_cast<cuuint64_t>(g.W) * cb, static_cast<cuuint64_t>(g.H * g.W) * cb};
        cuuint32_t box[4] = {static_cast<cuuint32_t>(a.sw), static_cast<cuuint32_t>(a.wv * a.stride),
                             static_cast<cuuint32_t>(a.rv * a.stride), 1};
        cuuint32_t es[4] = {1, static_cast<cuuint32_t>(a.stride), static_cast<cuuint32_t>(a.stride), 1};
        if (fn(mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t *>(xp), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

template <int CODE, int OUT, int SW, bool PAIRS>
cudaError_t launch_t(const CUtensorMap &ma, const CUtensorMap &mb, const ConvPlan &p, cudaStream_t s) {
    auto kern = conv_kernel<CODE, OUT, SW, PAIRS>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] { attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax); });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr = pdl_attribute();
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(p.smem);
    cfg.stream = s;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, p.a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int CODE, int SW>
cudaError_t launch_out(const CUtensorMap &ma, const CUtensorMap &mb, const ConvPlan &p, bt_dtype out_t,
                       cudaStream_t s) {
    switch (out_t) {
        case BT_F32: return launch_t<CODE, BT_F32, SW, false>(ma, mb, p, s);
        case BT_BF16:
            return p.a.pairs ? launch_t<CODE, BT_BF16, SW, true>(ma, mb, p, s)
                             : launch_t<CODE, BT_BF16, SW, false>(ma, mb, p, s);
        case BT_F16:
            return p.a.pairs ? launch_t<CODE, BT_F16, SW, true>(ma, mb, p, s)
                             : launch_t<CODE, BT_F16, SW, false>(ma, mb, p, s);
        default: return launch_t<CODE, BT_I32, SW, false>(ma, mb, p, s);
    }
}

}  // namespace

bool conv_implicit_applies(const ConvGeom &g, bt_code code) {
    if (const char *env = std::getenv("BT_CONV_IMPLICIT")) {
        if (std::strcmp(env, "0") == 0) return false;
    }
    ConvGeom q = g;
    q.O = kBM;                      // the plan's feasibility does not depend on O
    ConvPlan p;
    return plan_conv(q, code, 148, 4, p);   // 4-byte outputs need the most staging
}

cudaError_t launch_tc_conv_implicit(const uint8_t *xp, const uint8_t *wp, bt_code code, const ConvGeom &g, float alpha,
                                    void *out, bt_dtype out_t, unsigned int *err, cudaStream_t s,
                                    const float *scales) {
    if (!conv_implicit_applies(g, code)) return cudaErrorNotSupported;
    ConvPlan p;
    if (!plan_conv(g, code, device_sm_count(), out_t == BT_BF16 || out_t == BT_F16 ? 2 : 4, p))
        return cudaErrorNotSupported;
    p.a.alpha = alpha;
    p.a.scales = scales;
    p.a.out = out;
    p.a.err = err;
    p.a.wait_ns = wait_limit_ns();
    CUtensorMap ma, mb;
    if (!encode_maps(g, code, p.a, xp, wp, &ma, &mb)) return cudaErrorInvalidValue;
    if (code == BT_CODE_E4M3)
        return p.a.sw == 128 ? launch_out<BT_CODE_E4M3, 128>(ma, mb, p, out_t, s)
                             : launch_out<BT_CODE_E4M3, 64>(ma, mb, p, out_t, s);
    return p.a.sw == 128 ? launch_out<BT_CODE_E2M1, 128>(ma, mb, p, out_t, s)
                         : launch_out<BT_CODE_E2M1, 64>(ma, mb, p, out_t, s);
}

}  // namespace bt
