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
// Or the kernel packs x itself: six more warps read the tile's input rows of
// x (NCHW floats), shift and sign them, turn 32 pixels x 32 channels around
// with a bit-matrix transpose across the lanes and store each pixel's codes at
// its place in its phase image, swizzled as the copy would have left them. The
// convolution is then one kernel from x to y, and x is read once.
//
// Persistent, warp-specialised, one CTA per SM, single-CTA MMAs (M = 128):
//   warp 0 lane 0   TMA producer: the weights (resident for the whole launch
//                   when they fit beside two pixel stages, else a ring of
//                   slices re-read per tile) and a double-buffered stage of
//                   the tile's phase images (packed-pixel input only);
//   warp 1 lane 0   MMA issuer: per tap and K slice, the MMAs of its 32-byte K
//                   steps into the tile's accumulator buffer (double-buffered
//                   in TMEM, so a tile's epilogue overlaps the next tile's MMAs);
//   warps 2..9      epilogue, two per TMEM lane quarter (32 channels) taking
//                   alternate 32-column boxes: scale and cast, stage the box in
//                   shared memory, read it back with lanes along the pixels and
//                   store each channel's valid pixels (consecutive addresses of
//                   one NCHW plane per store instruction);
//   warps 10..15    (the kernel that packs x) the pixel stages from x, and
//                   the next tile's rows of x brought into L2 ahead.
// Every wait is bounded (bt_set_wait_timeout, 2 s by default; the teardown's
// drains of copies and MMAs in flight always 2 s): a wait that runs out
// records the timeout in the device error word and the kernel winds down
// without trapping.
//
// This header holds the kernel and its launch templates, shared by the
// translation units that instantiate it (packed-pixel input; one per float
// type of x for the kernel that packs x itself), so they compile in parallel.
#pragma once

#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "bt_device.cuh"
#include "bt_internal.h"
#include "sign_pack.cuh"
#include "tc_ptx.cuh"

namespace bt {
namespace conv {


constexpr int kBM = 128;                          // output channels per tile (MMA M)
constexpr int kEpiWarps = 8;
constexpr int kPackWarps = 6;                     // warps that pack x (the convolution that reads x itself)
template <bool FUSED> __host__ __device__ constexpr int conv_threads() {
    return 64 + 32 * kEpiWarps + (FUSED ? 32 * kPackWarps : 0);
}
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
    uint32_t tap[kMaxTaps];   // (tap index kh*k+kw << 24) | (phase << 20) | first staged row it reads
    uint32_t idesc;
    float alpha;
    const float *scales;      // not null: alpha = fp32(scales[0] * scales[1])
    void *out;                // NCHW [B, O, Ho, Wo]
    unsigned int *err;
    unsigned long long wait_ns;  // limit of each bounded wait of the main loops (teardown drains: kWaitNs)
    // the convolution that packs x itself (the pixel stages filled by the
    // packing warps instead of copies of packed pixels)
    const void *x;            // NCHW [B, C, H, W] floats (f32 / bf16 / f16)
    const float *bias;        // bias_a: one value, or one per input channel
    int bias_len;             // 0, 1 or C
    int C, H, W, HW;
    int ncg;                  // 32-channel groups of a packed pixel row (its bytes / code bytes of 32 channels)
    FastDiv div_w;            // division by W
    int ph_of[4];             // stride 2: phase image of (y mod 2, x mod 2), -1 where no tap reads; stride 1: 0
    int ph_ymin, ph_ymax;     // least and greatest ph_y0
    int zero_rows;            // more than one band per image: staged rows past the image are cleared per tile
    int prefetch;             // bring the next tile's image into L2 ahead (one band per image only)
    int a_early;              // resident weights may be copied before the wait for the previous kernel
                              // (set only when that kernel is the library's own pack of x)
    int ht2;                  // rows of a band per CTA (a pair: ht / 2 each; one CTA: ht)
    int nb;                   // accumulator columns per CTA's rows (a pair: bn / 2; one CTA: bn)
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

// CTA pair (cta_group::2): this CTA's copy into its own shared memory,
// completing on an mbarrier of either CTA of the pair (a shared::cluster
// address).
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap *m, int c0, int c1, int c2, int c3,
                                                 uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
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

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Bring `bytes` (a multiple of 16, from a 16-byte-aligned address) into L2.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Where the 128- / 64-byte swizzle puts a byte of shared memory: its 16-byte
// chunk index within the row XORed with the low bits of the row index
// (address bits 7..9 or 7..8), as the copies write it and the MMA reads it.
template <int SW> __device__ __forceinline__ uint32_t swizzled(uint32_t addr) {
    return addr ^ (((addr >> 7) & (SW == 128 ? 7u : 3u)) << 4);
}

__device__ __forceinline__ int sel4(const int (&v)[4], int i) {
    return i == 0 ? v[0] : (i == 1 ? v[1] : (i == 2 ? v[2] : v[3]));
}

// The units of one tile that one packing warp converts: a contiguous run
// [u0, u1) of (32-channel group cg, 32-pixel block blk), channel groups
// fastest. CHAN: a shift per channel (thresholds per load group) instead of
// one for all. Two units are in flight: the next unit's loads go out before
// the current one is converted.
struct PackTile {
    const uint8_t *xb;        // this image's planes
    int pa, plo, pe, r0;      // first pixel of block 0; the tile's pixel range; first output row
    uint32_t stage;           // the pixel stage being filled
};

template <typename XT, int CODE, int SW, bool CHAN>
__device__ __forceinline__ void pack_units(const ConvArgs &a, const PackTile &pt, int u0, int u1, int lane,
                                           uint32_t t_all, const int (&py0)[kMaxPhases], const int (&px0)[kMaxPhases],
                                           const int (&phof)[4]) {
    constexpr int OB = CODE == BT_CODE_E2M1 ? 16 : 32;          // code bytes of 32 channels
    constexpr int NV = sizeof(XT) == 2 ? 1 : 2;                 // 16-byte loads per 8 pixels
    constexpr int kLogSW = SW == 128 ? 7 : 6;
    const int C = a.C, HW = a.HW, W = a.W, ncg = a.ncg, s = a.stride, sh = a.stride - 1;
    const int rv = a.rv, wv = a.wv, nsl = a.nsl;
    const uint32_t img = a.img_bytes;
    const int lc = lane >> 2, lp = 8 * (lane & 3);
    // element offsets within the image: this lane's channel and pixel, and one load group further
    const uint32_t lane_off = static_cast<uint32_t>(lc) * HW + static_cast<uint32_t>(pt.pa + lp);
    const uint32_t grp = 8u * static_cast<uint32_t>(HW), cgs = 32u * static_cast<uint32_t>(HW);
    const XT *const xb = reinterpret_cast<const XT *>(pt.xb);
    // per-lane constants of the exchange rounds and the final shuffle
    const uint32_t keep16 = (lane & 16) ? 0xFFFF0000u : 0x0000FFFFu;
    const uint32_t keep8 = (lane & 8) ? 0xFF00FF00u : 0x00FF00FFu, rot8 = (lane & 8) ? 8u : 24u;
    const uint32_t keep4 = (lane & 4) ? 0xF0F0F0F0u : 0x0F0F0F0Fu, rot4 = (lane & 4) ? 4u : 28u;
    const int src_lane = ((lane & 1) << 4) | (((lane >> 2) & 1) << 3) | (((lane >> 1) & 1) << 2) |
                         (((lane >> 4) & 1) << 1) | ((lane >> 3) & 1);

    auto load = [&](uint4 (&g)[4][NV], int cg, int blk) {
        const uint32_t off = lane_off + static_cast<uint32_t>(cg) * cgs + 32u * static_cast<uint32_t>(blk);
        const int px = pt.pa + 32 * blk + lp;
        const int lim = C - cg * 32 - lc;
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int v = 0; v < NV; ++v)
                g[k][v] = ld_nc_v4_if(xb + off + k * grp + 4 * v, 8 * k < lim && px + 4 * v < HW);
    };
    // the place of this lane's pixel (after the transpose) for block blk
    bool store = false;
    uint32_t pix = 0, xpat = 0;
    auto place = [&](int blk) {
        const int p = pt.pa + 32 * blk + lane;
        const int y = static_cast<int>(fdiv(static_cast<uint32_t>(p), a.div_w));
        const int xx = p - y * W;
        const int ph = s == 1 ? 0 : sel4(phof, ((y & 1) << 1) | (xx & 1));
        const int phc = ph < 0 ? 0 : ph;
        const int r = ((y - sel4(py0, phc)) >> sh) - pt.r0;            // exact: y = ph_y0 (mod s)
        const int u = (xx - sel4(px0, phc)) >> sh;
        store = p >= pt.plo && p < pt.pe && ph >= 0 && static_cast<unsigned>(r) < static_cast<unsigned>(rv) &&
                static_cast<unsigned>(u) < static_cast<unsigned>(wv);
        pix = pt.stage + static_cast<uint32_t>(phc * nsl) * img + static_cast<uint32_t>(r * wv + u) * SW;
        xpat = ((pix >> 7) & (SW == 128 ? 7u : 3u)) << 4;             // the row's swizzle pattern
    };
    auto convert = [&](const uint4 (&g)[4][NV], int cg) {
        uint32_t w = 0;
        if constexpr (CODE == BT_CODE_E2M1) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t tk = t_all;
                if constexpr (CHAN) {
                    const int c = cg * 32 + 8 * k + lc;
                    tk = shift_threshold<XT>(c < C ? __ldg(a.bias + c) : 0.0f);
                }
                w |= sign_bits<XT>(g[k][0], g[k][NV - 1], tk, k);
            }
            w = exchange_rot(w, 16, keep16, 16u);
            w = exchange_rot(w, 8, keep8, rot8);
            w = exchange_rot(w, 4, keep4, rot4);
            w = __shfl_sync(0xFFFFFFFFu, w, src_lane);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int c = cg * 32 + 8 * k + lc;
                const float bc = a.bias_len > 1 ? (c < C ? __ldg(a.bias + c) : 0.0f) : (a.bias_len == 1 ? __ldg(a.bias) : 0.0f);
                Group<XT> gr;
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    gr.w[4 * v] = g[k][v].x; gr.w[4 * v + 1] = g[k][v].y;
                    gr.w[4 * v + 2] = g[k][v].z; gr.w[4 * v + 3] = g[k][v].w;
                }
                uint32_t P0, P1;
                if (isfinite(bc)) {
                    masks_ge<XT>(gr, -bc, P0, P1);
                } else {
                    float f[8], bb[8];
                    gr.unpack(f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) bb[e] = bc;
                    masks_add(f, bb, P0, P1);
                }
                w |= mask_byte(P0, P1) << (8 * k);
            }
            // lane bits (c2 c1 c0 p4 p3), register bits (c4 c3 p2 p1 p0) -> lane p, bit c
            w = exchange_bits<16, 4, 0x0F0F0F0Fu>(w, lane);
            w = exchange_bits<8, 2, 0x33333333u>(w, lane);
            w = exchange_bits<4, 1, 0x55555555u>(w, lane);
            w = __shfl_sync(0xFFFFFFFFu, w, ((lane & 7) << 2) | (lane >> 3));
        }
        if (!store) return;
        const int nvalid = C - cg * 32;
        const uint32_t o = static_cast<uint32_t>(cg * OB);
        // the chunk's place: its slice's image, its 16-byte chunk swizzled within the row
        const uint32_t addr = pix + (o >> kLogSW) * img + ((o & (SW - 1)) ^ xpat);
        if constexpr (CODE == BT_CODE_E2M1) {
            uint32_t qd[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) qd[i] = ((~w << (3 - i)) & 0x88888888u) | 0x22222222u;
            if (nvalid < 32) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int nv = nvalid - 8 * i;        // channels of this word inside C
                    if (nv < 8) qd[i] &= nv <= 0 ? 0u : (1u << (4 * nv)) - 1u;
                }
            }
            st_shared_v4(addr, qd[0], qd[1], qd[2], qd[3]);
        } else {
            // E4M3: +1 = 0x38, -1 = 0xB8, padding 0
            const uint32_t valid = nvalid >= 32 ? 0xFFFFFFFFu : (nvalid > 0 ? (1u << nvalid) - 1u : 0u);
            const uint32_t neg = ~w & valid;
            uint32_t qd[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t nb = (neg >> (8 * i)) & 0xFFu, vb = (valid >> (8 * i)) & 0xFFu;
                uint64_t v = 0x3838383838383838ull | (spread_bytes(nb) << 7);
                if (vb != 0xFFu) v &= spread_bytes(vb) * 0xFFull;
                qd[2 * i] = static_cast<uint32_t>(v);
                qd[2 * i + 1] = static_cast<uint32_t>(v >> 32);
            }
            st_shared_v4(addr, qd[0], qd[1], qd[2], qd[3]);
            st_shared_v4(addr ^ 16u, qd[4], qd[5], qd[6], qd[7]);   // the next chunk: xpat leaves bit 4 to o
        }
    };
    if (u0 >= u1) return;
    int cg = u0 % ncg, blk = u0 / ncg;
    place(blk);
    uint4 g0[4][NV], g1[4][NV];
    load(g0, cg, blk);
    for (int u = u0; u < u1; u += 2) {
        // unit u in g0, unit u + 1 (if any) into g1
        int cg1 = cg + 1, blk1 = blk;
        if (cg1 == ncg) { cg1 = 0; ++blk1; }
        const bool more = u + 1 < u1;
        if (more) load(g1, cg1, blk1);
        convert(g0, cg);
        if (!more) break;
        int cg2 = cg1 + 1, blk2 = blk1;
        if (cg2 == ncg) { cg2 = 0; ++blk2; }
        if (u + 2 < u1) load(g0, cg2, blk2);
        if (blk1 != blk) place(blk1);
        convert(g1, cg1);
        if (blk2 != blk1 && u + 2 < u1) place(blk2);
        cg = cg2;
        blk = blk2;
    }
}

// Pack the tiles' pixels from x straight into the pixel stages: the same bytes
// the copies of packed NHWC pixels would put there (the shift + sign of
// bitorch-engine BinaryConv2dCutlass.set_activation, then the channel
// packing). A unit is (32 channels, 32 consecutive pixels of the tile's input
// rows); each warp takes a contiguous run of the tile's units, channel groups
// fastest, so a pixel's place in the stage is worked out once per block of 32
// pixels. Lane l loads 8 pixels (16 bytes of a 2-byte type, 32 of f32) of
// channel 32 cg + 8 k + l / 4, k = 0..3, as predicated loads; the sign bits
// start at lane bits (c2 c1 c0 p4 p3) and register bits (p0 p2 p1 c4 c3);
// three exchange rounds (lane bits c2, c1, c0 against register bits p0, p2,
// p1) and one shuffle leave lane p with register bits (c2 c1 c0 c4 c3):
// channel c at bit 4 (c % 8) + c / 8, so the E2M1 codes of channels 8i..8i+7
// (+1 = 0x2, -1 = 0xA, channel 8i + j in nibble j) are one shift and one
// logic op: ((~w << (3 - i)) & 0x88888888) | 0x22222222. E4M3 codes (+1 =
// 0x38, -1 = 0xB8) take the natural channel order instead. Consecutive lanes
// end on consecutive pixels, so each 16-byte store instruction (two for E4M3)
// spreads over the banks. Pixels no tap reads, or outside the staged rows,
// are dropped; staged places no input pixel reaches keep the zeros they were
// given.
template <typename XT, int CODE, int SW, bool CP>
__device__ __forceinline__ void pack_tiles(const ConvArgs &a, uint32_t sB, uint32_t bars, int pw, int lane,
                                           volatile uint32_t *abort_flag, int unit, int nunits, int row_first,
                                           bool leader) {
    constexpr int kPT = kPackWarps * 32;
    const XT *const x = static_cast<const XT *>(a.x);
    const int s = a.stride;
    const int C = a.C, H = a.H, W = a.W, HW = a.HW;
    const int rv = a.rv, ncg = a.ncg, nsl = a.nsl, nph = a.nph, ht = a.ht;
    const int num_ot = a.num_ot, bands = a.bands, num_tiles = a.num_tiles;
    const uint32_t img = a.img_bytes, stage_bytes = a.stage_bytes;
    int py0[kMaxPhases], px0[kMaxPhases], phof[4];
#pragma unroll
    for (int i = 0; i < kMaxPhases; ++i) {
        py0[i] = a.ph_y0[i];
        px0[i] = a.ph_x0[i];
        phof[i] = a.ph_of[i];
    }
    auto bfull = [&](int i) { return bars + 8u * (2 * kMaxAStages + i); };
    auto bempty = [&](int i) { return bars + 8u * (2 * kMaxAStages + 2 + i); };
    // input rows [ylo, yhi] of the tile starting at output row r0 (empty: ylo > yhi)
    auto rows_of = [&](int r0, int &ylo, int &yhi) {
        ylo = s * r0 + a.ph_ymin;
        yhi = s * (r0 + rv - 1) + a.ph_ymax;
        if (ylo < 0) ylo = 0;
        if (yhi > H - 1) yhi = H - 1;
    };
    // warp 0: a tile that reads whole channel planes (one band per image)
    // brings its image into L2 ahead, in 32 KB requests (the copy engine's cost
    // is per request); other tiles are not prefetched
    auto prefetch_tile = [&](int t) {
        const int b = (t / num_ot) / bands;
        const uint64_t total = static_cast<uint64_t>(C) * HW * sizeof(XT);
        const uint8_t *base = reinterpret_cast<const uint8_t *>(x + static_cast<int64_t>(b) * C * HW);
        for (uint64_t o = static_cast<uint64_t>(lane) << 15; o < total; o += uint64_t(32) << 15) {
            const uint64_t n = total - o < (uint64_t(1) << 15) ? total - o : (uint64_t(1) << 15);
            prefetch_l2(base + o, static_cast<uint32_t>(n));
        }
    };
    const bool prefetch = a.prefetch != 0 && bands == 1 && leader;

    pdl_wait();                                       // x (and bias) may come from the previous kernel
    const uint32_t t_all = shift_threshold<XT>(a.bias_len == 1 ? __ldg(a.bias) : 0.0f);
    const bool chan = a.bias_len > 1;
    if (prefetch && pw == 0 && unit < num_tiles) prefetch_tile(unit);
    // both pixel stages start cleared: staged places that no input pixel
    // reaches (the padding around the image) keep code 0 for the whole launch
    {
        const uint32_t n16 = (static_cast<uint32_t>(a.b_stages) * stage_bytes) >> 4;
        for (uint32_t i = static_cast<uint32_t>(pw * 32 + lane); i < n16; i += kPT) st_shared_v4(sB + 16u * i, 0u, 0u, 0u, 0u);
        asm volatile("bar.sync 1, %0;" ::"r"(kPT) : "memory");
    }
    const uint32_t rowb = static_cast<uint32_t>(a.wv) * a.sw;  // bytes of one staged row of one slice
    int bs = 0;
    uint32_t bph = 0;
    for (int t = unit; t < num_tiles; t += nunits) {
        const int rest = t / num_ot;
        const int b = rest / bands, band = rest - b * bands;
        const int r0 = band * ht + row_first;             // this CTA's first row of the band
        if (prefetch && pw == 0 && t + nunits < num_tiles) prefetch_tile(t + nunits);
        if (!tc::wait_fast(bempty(bs), bph ^ 1u, abort_flag, a.err, a.wait_ns)) break;
        const uint32_t stage = sB + static_cast<uint32_t>(bs) * stage_bytes;
        if (a.zero_rows) {
            // staged rows above or below the image: a tile of another band may have filled them
            for (int i = pw; i < nph * rv; i += kPackWarps) {
                const int ph = i / rv, r = i - ph * rv;
                const int y = s * (r0 + r) + sel4(py0, ph);
                if (y >= 0 && y < H) continue;
                for (int sl = 0; sl < nsl; ++sl) {
                    const uint32_t row0 = stage + static_cast<uint32_t>(ph * nsl + sl) * img + static_cast<uint32_t>(r) * rowb;
                    for (uint32_t o = static_cast<uint32_t>(lane) * 16u; o < rowb; o += 512u)
                        st_shared_v4(row0 + o, 0u, 0u, 0u, 0u);
                }
            }
        }
        int ylo, yhi;
        rows_of(r0, ylo, yhi);
        if (ylo <= yhi) {
            PackTile pt;
            pt.plo = ylo * W;
            pt.pe = (yhi + 1) * W;
            pt.pa = pt.plo & ~31;                         // 32-pixel blocks from an aligned start
            pt.r0 = r0;
            pt.stage = stage;
            pt.xb = reinterpret_cast<const uint8_t *>(x + static_cast<int64_t>(b) * C * HW);
            const int units = ((pt.pe - pt.pa + 31) >> 5) * ncg;
            // this warp's contiguous run of units [u0, u1), channel groups fastest
            const int u0 = (units * pw) / kPackWarps, u1 = (units * (pw + 1)) / kPackWarps;
            if (chan) pack_units<XT, CODE, SW, true>(a, pt, u0, u1, lane, t_all, py0, px0, phof);
            else pack_units<XT, CODE, SW, false>(a, pt, u0, u1, lane, t_all, py0, px0, phof);
        }
        // make the stage's generic-proxy writes visible to the tensor core
        // (of both CTAs of a pair: the arrival is on the even CTA's barrier)
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (CP && !leader) tc::mbar_arrive_cluster(tc::mapa(bfull(bs), 0u));
            else tc::mbar_arrive(bfull(bs));
        }
        if (++bs == a.b_stages) { bs = 0; bph ^= 1u; }
    }
}

// XT = void: the pixel stages are copies of packed NHWC pixels (tmB); XT = the
// input's float type: the packing warps fill them from x (tmB unused).
// CP: a cluster of two CTAs computes 256-channel tiles with cta_group::2 MMAs
// (M = 256): CTA r holds the weights of channels [256 ot + 128 r, + 128) and
// the pixels of rows [r ht2, (r + 1) ht2) of the band (plus the taps' reach),
// N / 2 = nb accumulator columns each; the even CTA issues the MMAs, every
// copy, pack and epilogue hand-off completes on its barriers, and its commits
// reach both CTAs.
template <int CODE, int OUT, int SW, bool PAIRS, typename XT, bool CP>
__global__ void __launch_bounds__(conv_threads<!std::is_void<XT>::value>(), 1)
conv_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const __grid_constant__ ConvArgs a) {
    constexpr bool kFused = !std::is_void<XT>::value;
    using T = typename OutT<OUT>::type;
    constexpr int kElem = sizeof(T);
    constexpr int kBoxRow = 32 * kElem;              // bytes of one staging-box row
    constexpr uint32_t kASlice = kBM * SW;           // weight bytes per K slice
    constexpr int kMmaPerSlice = SW / 32;            // 32 bytes of K per MMA
    constexpr uint32_t kAccStride = CODE == BT_CODE_E2M1 ? 240u : 256u;
    constexpr uint32_t kPeers = CP ? 2u : 1u;
    constexpr int kEpiBatch = kFused ? 1 : 2;         // TMEM boxes loaded per wait (registers: 32 per box)

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
    const uint32_t crank = CP ? tc::cluster_ctarank() : 0u;
    const bool leader = !CP || crank == 0;
    // a barrier of the even CTA, as this CTA addresses it
    auto lead = [&](uint32_t bar) { return CP ? tc::mapa(bar, 0u) : bar; };
    if (threadIdx.x == 0) pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < kMaxAStages; ++i) {
            tc::mbar_init(afull(i), 1);
            tc::mbar_init(aempty(i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bfull(i), kFused ? kPeers * kPackWarps : 1u);
            tc::mbar_init(bempty(i), 1);
            tc::mbar_init(tfull(i), 1);
            tc::mbar_init(tempty(i), kPeers * kEpiWarps);
        }
        tc::mbar_init(drain, 1);
        *abort_flag = 0u;
        tc::fence_mbar_init();
        tc::prefetch_map(&tmA);
        if (!kFused) tc::prefetch_map(&tmB);
    }
    if (warp == 1) {
        if (CP) {
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
    const int quarter = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    if (CODE == BT_CODE_E2M1 && warp >= 2 && warp < 6) {
        tc::tmem_st16_fill(tmem + lane_base + kSfCol, kUnitScales);
        tc::tmem_st16_fill(tmem + lane_base + kSfCol + 16, kUnitScales);
        tc::tmem_st_wait();
    }
    tc::fence_before_sync();
    __syncthreads();
    // the peer's barriers and block scales exist before any copy, commit or MMA reaches them
    if (CP) tc::cluster_sync();
    tc::fence_after_sync();

    const int unit = CP ? static_cast<int>(tc::cluster_id_x()) : static_cast<int>(blockIdx.x);
    const int nunits = CP ? static_cast<int>(tc::num_clusters_x()) : static_cast<int>(gridDim.x);
    const int hw = a.Ho * a.Wo;
    const int row_first = static_cast<int>(crank) * a.ht2;   // this CTA's first row of a band
    const int ch_first = static_cast<int>(crank) * kBM;      // this CTA's first channel of a tile

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int as = 0, bs = 0;
            uint32_t aph = 0, bph = 0;
            uint32_t a_last[kMaxAStages], b_last[2];      // phase of each slot's last copy; 2 = none
            for (int i = 0; i < kMaxAStages; ++i) a_last[i] = 2u;
            b_last[0] = b_last[1] = 2u;
            bool ok = true, a_loaded = false;
            // resident weights: one barrier per box (up to kMaxAStages boxes; more
            // share the first barrier), so that the first MMAs start once their
            // taps have landed
            auto load_weights = [&](int ot) {
                const int am0 = ot * static_cast<int>(kPeers) * kBM + ch_first;
                const bool per_box = a.a_boxes <= kMaxAStages;
                if (!per_box && leader)
                    tc::mbar_arrive_expect_tx(afull(0), kPeers * static_cast<uint32_t>(a.a_boxes * a.a_d) * kASlice);
                for (int i = 0; i < a.a_boxes; ++i) {
                    const int bi = per_box ? i : 0;
                    if (per_box && leader) tc::mbar_arrive_expect_tx(afull(i), kPeers * static_cast<uint32_t>(a.a_d) * kASlice);
                    if (per_box) a_last[i] = 0u;
                    const uint32_t dst = sA + static_cast<uint32_t>(i * a.a_d) * kASlice;
                    if (CP) tc::tma_load_3d_pair(dst, &tmA, 0, am0, i * a.a_d, lead(afull(bi)));
                    else tc::tma_load_3d(dst, &tmA, 0, am0, i * a.a_d, afull(bi));
                }
                if (!per_box) a_last[0] = 0u;
                a_loaded = true;
            };
            // the weights are not written by the library's own pack of x, which is
            // the kernel this one may overlap: they can be in flight before the wait
            if (a.a_resident && a.a_early && unit < a.num_tiles) load_weights(unit % a.num_ot);
            pdl_wait();                                   // pixels (and otherwise weights) come from earlier kernels
            for (int t = unit; t < a.num_tiles && ok; t += nunits) {
                const int ot = t % a.num_ot, rest = t / a.num_ot;
                const int b = rest / a.bands, band = rest - b * a.bands;
                const int r0 = band * a.ht + row_first;
                const int am0 = ot * static_cast<int>(kPeers) * kBM + ch_first;
                // the tile's phase images (the packing warps fill them from x instead)
                if (!kFused) {
                    if (!tc::wait_fast(bempty(bs), bph ^ 1u, abort_flag, a.err, a.wait_ns)) { ok = false; break; }
                    if (leader) tc::mbar_arrive_expect_tx(bfull(bs), kPeers * static_cast<uint32_t>(a.nph * a.nsl) * a.img_tx);
                    const uint32_t dst0 = sB + static_cast<uint32_t>(bs) * a.stage_bytes;
                    const uint32_t fbar = lead(bfull(bs));
                    for (int ph = 0; ph < a.nph; ++ph)
                        for (int sl = 0; sl < a.nsl; ++sl) {
                            const uint32_t dst = dst0 + static_cast<uint32_t>(ph * a.nsl + sl) * a.img_bytes;
                            if (CP) tma_load_4d_pair(dst, &tmB, sl * SW, a.ph_x0[ph], a.stride * r0 + a.ph_y0[ph], b, fbar);
                            else tma_load_4d(dst, &tmB, sl * SW, a.ph_x0[ph], a.stride * r0 + a.ph_y0[ph], b, fbar);
                        }
                    b_last[bs] = bph;
                    if (++bs == a.b_stages) { bs = 0; bph ^= 1u; }
                }
                // resident weights (unless already in flight): after the first tile's pixels
                if (a.a_resident && !a_loaded) load_weights(ot);
                if (!a.a_resident) {
                    for (int i0 = 0; i0 < nslices; i0 += a.a_d) {
                        if (!tc::wait_fast(aempty(as), aph ^ 1u, abort_flag, a.err, a.wait_ns)) { ok = false; break; }
                        if (leader) tc::mbar_arrive_expect_tx(afull(as), kPeers * static_cast<uint32_t>(a.a_d) * kASlice);
                        const uint32_t dst = sA + static_cast<uint32_t>(as * a.a_d) * kASlice;
                        if (CP) tc::tma_load_3d_pair(dst, &tmA, 0, am0, i0, lead(afull(as)));
                        else tc::tma_load_3d(dst, &tmA, 0, am0, i0, afull(as));
                        a_last[as] = aph;
                        if (++as == a.a_stages) { as = 0; aph ^= 1u; }
                    }
                }
            }
            if (!ok && leader) {
                // let every issued copy land before the CTA can exit (a pair's
                // copies all complete on the even CTA's barriers)
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
        if (lane == 0 && leader) {
            // ---------------- MMA issuer ----------------
            int as = 0, bs = 0, local = 0;
            uint32_t aph = 0, bph = 0;
            bool ok = true;
            // Up to kRegTaps taps of one K slice each with resident weights: every
            // tap's A descriptor and B offset is built once, in registers, so a
            // tile's MMAs go out back to back (building a tap's descriptors at issue
            // time measured ~50 % slower per MMA on GB300 for 64-byte slices).
            constexpr int kRegTaps = 9;
            const bool reg_taps = a.a_resident && a.nsl == 1 && a.ntap <= kRegTaps;
            const uint64_t adesc_base0 = kmajor_desc(sA, SW);
            uint64_t adesc_t[kRegTaps];
            uint32_t boff_t[kRegTaps];
#pragma unroll
            for (int t = 0; t < kRegTaps; ++t) {
                const uint32_t tapw = t < a.ntap ? a.tap[t] : 0u;
                adesc_t[t] = adesc_base0 + static_cast<uint64_t>(tapw >> 24) * ((kBM * SW) >> 4);
                boff_t[t] = ((tapw >> 20) & 0xFu) * (a.img_bytes >> 4) + (tapw & 0xFFFFFu) * (SW >> 4);
            }
            for (int t = unit; t < a.num_tiles && ok; t += nunits, ++local) {
                const int buf = local & 1;
                if (local >= 2) {
                    // the epilogue (of both CTAs of a pair) has drained this buffer
                    if (!tc::wait_fast(tempty(buf), static_cast<uint32_t>((local - 2) >> 1) & 1u, abort_flag, a.err, a.wait_ns))
                        break;
                    tc::fence_after_sync();
                }
                if (!tc::wait_fast(bfull(bs), bph, abort_flag, a.err, a.wait_ns)) break;
                tc::fence_after_sync();
                const uint32_t dacc = tmem + static_cast<uint32_t>(buf) * kAccStride;
                if (reg_taps) {
                    const uint64_t bbase = kmajor_desc(sB + static_cast<uint32_t>(bs) * a.stage_bytes, SW);
                    uint64_t bdt[kRegTaps];
#pragma unroll
                    for (int t = 0; t < kRegTaps; ++t) bdt[t] = bbase + boff_t[t];
                    uint32_t waited = 0;                  // first tile: weight boxes already waited for
#pragma unroll
                    for (int t = 0; t < kRegTaps; ++t) {
                        if (t < a.ntap) {
                            if (local == 0) {
                                const int bx = a.a_boxes <= kMaxAStages ? static_cast<int>(a.tap[t] >> 24) / a.a_d : 0;
                                if (!((waited >> bx) & 1u)) {
                                    if (!tc::wait_fast(afull(bx), 0u, abort_flag, a.err, a.wait_ns)) { ok = false; break; }
                                    tc::fence_after_sync();
                                    waited |= 1u << bx;
                                }
                            }
#pragma unroll
                            for (int kk = 0; kk < kMmaPerSlice; ++kk) {
                                const uint32_t acc = (t | kk) != 0 ? 1u : 0u;
                                if (CP) {
                                    if (CODE == BT_CODE_E4M3) tc::mma_f8f6f4_pair(dacc, adesc_t[t] + 2 * kk, bdt[t] + 2 * kk, a.idesc, acc);
                                    else tc::mma_mxf4_pair(dacc, adesc_t[t] + 2 * kk, bdt[t] + 2 * kk, a.idesc, tmem + kSfCol, tmem + kSfCol + 16, acc);
                                } else {
                                    if (CODE == BT_CODE_E4M3) tc::mma_f8f6f4(dacc, adesc_t[t] + 2 * kk, bdt[t] + 2 * kk, a.idesc, acc);
                                    else tc::mma_mxf4(dacc, adesc_t[t] + 2 * kk, bdt[t] + 2 * kk, a.idesc, tmem + kSfCol, tmem + kSfCol + 16, acc);
                                }
                            }
                        }
                    }
                } else {
                // descriptors are built once and moved by adding (byte offset >> 4)
                // to their start-address field (shared-memory addresses stay below
                // 256 KB, so the 14-bit field never carries): the issuing thread
                // spends a few integer adds per MMA, not a descriptor build
                const uint64_t bdesc_stage = kmajor_desc(sB + static_cast<uint32_t>(bs) * a.stage_bytes, SW);
                const uint64_t adesc_base = kmajor_desc(sA, SW);
                const uint32_t img16 = a.img_bytes >> 4;
                constexpr uint32_t kSlice16 = kASlice >> 4;
                uint64_t adesc = adesc_base;
                int idx = 0, within = 0;
                uint32_t waited = 0;                      // first tile: weight boxes already waited for
                for (int tp = 0; tp < a.ntap && ok; ++tp) {
                    // each tap: its phase image, its first staged row, its own weight slices
                    const uint32_t tapw = a.tap[tp];
                    const int tap_id = static_cast<int>(tapw >> 24);
                    uint64_t bd = bdesc_stage + ((tapw >> 20) & 0xFu) * static_cast<uint32_t>(a.nsl) * img16 +
                                  (tapw & 0xFFFFFu) * (SW >> 4);
                    for (int sl = 0; sl < a.nsl; ++sl, ++idx) {
                        if (a.a_resident) {
                            const int sidx = tap_id * a.nsl + sl;           // the slice's place in the resident weights
                            if (local == 0) {
                                // first tile: the box of weights holding this slice (each box on its own
                                // barrier, or all on the first)
                                const int bx = a.a_boxes <= kMaxAStages ? sidx / a.a_d : 0;
                                if (!((waited >> bx) & 1u)) {
                                    if (!tc::wait_fast(afull(bx), 0u, abort_flag, a.err, a.wait_ns)) { ok = false; break; }
                                    tc::fence_after_sync();
                                    waited |= 1u << bx;
                                }
                            }
                            adesc = adesc_base + static_cast<uint64_t>(sidx) * kSlice16;
                        } else if (within == 0) {
                            if (!tc::wait_fast(afull(as), aph, abort_flag, a.err, a.wait_ns)) { ok = false; break; }
                            tc::fence_after_sync();
                            adesc = adesc_base + static_cast<uint64_t>(as * a.a_d) * kSlice16;
                        }
#pragma unroll
                        for (int kk = 0; kk < kMmaPerSlice; ++kk) {
                            const uint32_t acc = (idx | kk) != 0 ? 1u : 0u;
                            if (CP) {
                                if (CODE == BT_CODE_E4M3) tc::mma_f8f6f4_pair(dacc, adesc + 2 * kk, bd + 2 * kk, a.idesc, acc);
                                else tc::mma_mxf4_pair(dacc, adesc + 2 * kk, bd + 2 * kk, a.idesc, tmem + kSfCol, tmem + kSfCol + 16, acc);
                            } else {
                                if (CODE == BT_CODE_E4M3) tc::mma_f8f6f4(dacc, adesc + 2 * kk, bd + 2 * kk, a.idesc, acc);
                                else tc::mma_mxf4(dacc, adesc + 2 * kk, bd + 2 * kk, a.idesc, tmem + kSfCol, tmem + kSfCol + 16, acc);
                            }
                        }
                        adesc += kSlice16;
                        bd += img16;
                        if (++within == a.a_d) {
                            within = 0;
                            if (!a.a_resident) {
                                if (CP) tc::mma_commit_pair(aempty(as), 0x3);
                                else tc::mma_commit(aempty(as));
                                if (++as == a.a_stages) { as = 0; aph ^= 1u; }
                            }
                        }
                    }
                }
                }
                if (!ok) break;
                if (CP) {
                    tc::mma_commit_pair(bempty(bs), 0x3);
                    tc::mma_commit_pair(tfull(buf), 0x3);
                } else {
                    tc::mma_commit(bempty(bs));
                    tc::mma_commit(tfull(buf));
                }
                if (++bs == a.b_stages) { bs = 0; bph ^= 1u; }
            }
            // every MMA issued must finish before the accumulator is freed
            if (CP) tc::mma_commit_pair(drain, 0x1);
            else tc::mma_commit(drain);
            const unsigned long long t0 = globaltimer_ns();
            while (!tc::mbar_try_wait(drain, 0u) && globaltimer_ns() - t0 < kWaitNs) {}
        }
        __syncwarp();
    } else if (kFused && warp >= 2 + kEpiWarps) {
        // ---------------- packing warps (10..15) ----------------
        if constexpr (kFused)
            pack_tiles<XT, CODE, SW, CP>(a, sB, bars, warp - 2 - kEpiWarps, lane, abort_flag, unit, nunits, row_first, leader);
    } else {
        // ---------------- epilogue (warps 2..9) ----------------
        pdl_wait();                                       // the previous kernel may still use `out`
        T *const out = static_cast<T *>(a.out);
        const uint32_t sbox = sStage + static_cast<uint32_t>((warp - 2) * 32 * 32 * kElem);
        const float alpha = a.scales != nullptr ? alpha_from(a.scales) : a.alpha;
        const int half = (warp - 2) / 4;
        // accumulator column -> virtual pixel of the band: the second half (a
        // pair's odd CTA) starts at row ht2, its columns at nb
        const int hcols = a.ht2 * a.wv, vshift = hcols - a.nb;
        int local = 0;
        for (int t = unit; t < a.num_tiles; t += nunits, ++local) {
            const int ot = t % a.num_ot, rest = t / a.num_ot;
            const int b = rest / a.bands, band = rest - b * a.bands;
            const int r0 = band * a.ht;
            const int hte = a.Ho - r0 < a.ht ? a.Ho - r0 : a.ht;       // output rows of this band
            const int buf = local & 1;
            if (!tc::wait_fast(tfull(buf), static_cast<uint32_t>(local >> 1) & 1u, abort_flag, a.err, a.wait_ns)) break;
            tc::fence_after_sync();
            const int o0 = ot * static_cast<int>(kPeers) * kBM + ch_first + quarter * 32;   // this warp's first channel
            const int nrows = a.O - o0 < 32 ? a.O - o0 : 32;
            const int ncols = hte * a.wv;
            const int nbox = CP ? (a.bn + 31) / 32 : (ncols + 31) / 32;
            const uint32_t tbase = tmem + lane_base + static_cast<uint32_t>(buf) * kAccStride;
            T *const plane0 = out + (static_cast<int64_t>(b) * a.O + o0) * hw + static_cast<int64_t>(r0) * a.Wo;
            // hand the accumulator back once every TMEM read of this tile is complete
            auto release = [&]() {
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if (CP && !leader) tc::mbar_arrive_cluster(tc::mapa(tempty(buf), 0u));
                    else tc::mbar_arrive(tempty(buf));
                }
            };
            if (nrows <= 0) {
                release();
            } else {
                // this warp's boxes bx = half, half + 2, ... in batches of kEpiBatch: the
                // TMEM loads of a batch go out together and are waited for once (a
                // load waits long while MMAs of the other buffer run, most under CTA
                // pairs); the accumulator goes back after the last batch's loads
                const int nmine = (nbox - half + 1) / 2;
                // a warp with no box of this tile (a band of at most 32 valid
                // columns) still hands the accumulator back
                if (nmine <= 0) release();
                for (int j0 = 0; j0 < nmine; j0 += kEpiBatch) {
                    uint32_t r[kEpiBatch][32];
#pragma unroll
                    for (int j = 0; j < kEpiBatch; ++j)
                        if (j0 + j < nmine) tc::tmem_ld32(tbase + static_cast<uint32_t>(32 * (half + 2 * (j0 + j))), r[j]);
                    tc::tmem_ld_wait();
                    if (j0 + kEpiBatch >= nmine) release();
#pragma unroll
                    for (int j = 0; j < kEpiBatch; ++j) {
                        if (j0 + j >= nmine) break;
                        const int bx = half + 2 * (j0 + j);
                        // stage: row = this lane's channel, 32 virtual pixels, swizzled
                        __syncwarp();
#pragma unroll
                        for (int q = 0; q < kBoxRow / 16; ++q) {
                            const uint32_t addr = sbox + static_cast<uint32_t>(lane * kBoxRow) + (box_chunk<kElem>(q, lane) << 4);
                            const uint4 w = chunk16<OUT, kElem>(r[j], q * (16 / kElem), alpha);
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w.x), "r"(w.y),
                                         "r"(w.z), "r"(w.w)
                                         : "memory");
                        }
                        __syncwarp();
                        // read back with lanes along the pixels
                        if constexpr (PAIRS) {
                            const int col = 32 * bx + 2 * (lane & 15);
                            const int sec = col >= a.nb ? 1 : 0;
                            const int v = col + sec * vshift;
                            const int i = v / a.wv, jx = v - i * a.wv;
                            const bool valid = col < a.bn && col - sec * a.nb < hcols && v < ncols && jx < a.Wo;
                            uint8_t *p = reinterpret_cast<uint8_t *>(plane0 + static_cast<int64_t>(lane >> 4) * hw +
                                                                     static_cast<int64_t>(i) * a.Wo + jx);
                            box_to_planes_pairs(sbox, lane, valid, p, static_cast<int64_t>(hw) * kElem, nrows);
                        } else {
                            const int col = 32 * bx + lane;            // lane = accumulator column
                            const int sec = col >= a.nb ? 1 : 0;
                            const int v = col + sec * vshift;
                            const int i = v / a.wv, jx = v - i * a.wv;
                            const bool valid = col < a.bn && col - sec * a.nb < hcols && v < ncols && jx < a.Wo;
                            uint8_t *p = reinterpret_cast<uint8_t *>(plane0 + static_cast<int64_t>(i) * a.Wo + jx);
                            box_to_planes<kElem>(sbox, lane, valid, p, static_cast<int64_t>(hw) * kElem, nrows);
                        }
                    }
                }
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    // no CTA of a pair leaves while its peer may still signal its barriers or
    // run MMAs on its shared memory and TMEM
    if (CP) tc::cluster_sync();
    if (warp == 1) {
        tc::fence_after_sync();
        if (CP) tc::tmem_dealloc_pair(tmem, kTmemCols);
        else tc::tmem_dealloc(tmem, kTmemCols);
    }
}

struct ConvPlan {
    ConvArgs a;
    bool cp;                  // CTA pairs (clusters of two, cta_group::2 MMAs)
    int smem;
    int grid;
};

template <int CODE, int OUT, int SW, bool PAIRS, typename XT, bool CP>
cudaError_t launch_cp(const CUtensorMap &ma, const CUtensorMap &mb, const ConvPlan &p, cudaStream_t s) {
    auto kern = conv_kernel<CODE, OUT, SW, PAIRS, XT, CP>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] { attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax); });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0] = pdl_attribute();
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CP ? 2 : 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid), 1, 1);
    cfg.blockDim = dim3(conv_threads<!std::is_void<XT>::value>(), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(p.smem);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = CP ? 2 : 1;
    if (CP) {
        // as many pairs as fit at once (one query per device and shared-memory
        // size); resident weights keep each pair on one channel tile
        static std::mutex mu;
        static int cached_smem[128] = {}, cached_fit[128] = {};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) dev = 0;
        int fit = 0;
        {
            std::lock_guard<std::mutex> lock(mu);
            if (cached_smem[dev] == p.smem) {
                fit = cached_fit[dev];
            } else {
                if (cudaOccupancyMaxActiveClusters(&fit, kern, &cfg) != cudaSuccess) fit = 0;
                cached_smem[dev] = p.smem;
                cached_fit[dev] = fit;
            }
        }
        int units = p.grid / 2;
        if (fit > 0 && fit < units) {
            units = p.a.a_resident ? fit / p.a.num_ot * p.a.num_ot : fit;
            if (units < 1) units = 1;
            cfg.gridDim = dim3(static_cast<unsigned>(2 * units), 1, 1);
        }
    }
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, p.a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int CODE, int OUT, int SW, bool PAIRS, typename XT>
cudaError_t launch_t(const CUtensorMap &ma, const CUtensorMap &mb, const ConvPlan &p, cudaStream_t s) {
    return p.cp ? launch_cp<CODE, OUT, SW, PAIRS, XT, true>(ma, mb, p, s)
                : launch_cp<CODE, OUT, SW, PAIRS, XT, false>(ma, mb, p, s);
}

template <int CODE, int SW, typename XT>
cudaError_t launch_out(const CUtensorMap &ma, const CUtensorMap &mb, const ConvPlan &p, bt_dtype out_t,
                       cudaStream_t s) {
    switch (out_t) {
        case BT_F32: return launch_t<CODE, BT_F32, SW, false, XT>(ma, mb, p, s);
        case BT_BF16:
            return p.a.pairs ? launch_t<CODE, BT_BF16, SW, true, XT>(ma, mb, p, s)
                             : launch_t<CODE, BT_BF16, SW, false, XT>(ma, mb, p, s);
        case BT_F16:
            return p.a.pairs ? launch_t<CODE, BT_F16, SW, true, XT>(ma, mb, p, s)
                             : launch_t<CODE, BT_F16, SW, false, XT>(ma, mb, p, s);
        default: return launch_t<CODE, BT_I32, SW, false, XT>(ma, mb, p, s);
    }
}

template <typename XT>
cudaError_t launch_code(const CUtensorMap &ma, const CUtensorMap &mb, const ConvPlan &p, bt_code code, bt_dtype out_t,
                        cudaStream_t s) {
    if (code == BT_CODE_E4M3)
        return p.a.sw == 128 ? launch_out<BT_CODE_E4M3, 128, XT>(ma, mb, p, out_t, s)
                             : launch_out<BT_CODE_E4M3, 64, XT>(ma, mb, p, out_t, s);
    return p.a.sw == 128 ? launch_out<BT_CODE_E2M1, 128, XT>(ma, mb, p, out_t, s)
                         : launch_out<BT_CODE_E2M1, 64, XT>(ma, mb, p, out_t, s);
}

// Instantiated one translation unit per input type: the convolution that packs
// x of that float type itself (the pixel-map slot takes the weights' map).
cudaError_t launch_fused_f32(const CUtensorMap &ma, const ConvPlan &p, bt_code code, bt_dtype out_t, cudaStream_t s);
cudaError_t launch_fused_bf16(const CUtensorMap &ma, const ConvPlan &p, bt_code code, bt_dtype out_t, cudaStream_t s);
cudaError_t launch_fused_f16(const CUtensorMap &ma, const ConvPlan &p, bt_code code, bt_dtype out_t, cudaStream_t s);

}  // namespace conv
}  // namespace bt
