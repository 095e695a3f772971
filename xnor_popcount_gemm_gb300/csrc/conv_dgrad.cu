// Input gradient of the binary conv2d layer's straight-through backward
// (bitorch-engine BinaryConv2dForward.backward):
//   grad_input = bf16(conv2d_input(x.shape, bf16(sign(w) * scale_w), g))
//                * !(q < -1 || q > 1),  q = x / scale_a in x's dtype
//   grad_scale_a = sum(grad_input * sign(x) / sqrt(numel(x)))
// as one implicit GEMM on the tensor cores: no tap matrix reaches memory.
//
// Sub-pixel phases. Input row h receives output row i through kernel row kh
// when h + p - kh*d = s*i. Writing h = s*m + rh (rh the row's phase), the
// rows kh with (rh + p - kh*d) divisible by s are the phase's taps, each at
// the fixed offset oh = (rh + p - kh*d) / s: i = m + oh. Columns likewise. So
// every phase (rh, rw) of the input gradient is a stride-1 correlation of g
// with its own taps:
//   gx[b, c, s*m + rh, s*n + rw] = bf16(scale_w) * sum over the phase's taps
//       (kh, kw) and o of sign(w)[o, c, kh, kw] * g[b, o, m + oh, n + ow]
// (g zero outside the output image), the phases together using each of the
// k*k taps once.
//
// Tiles. M = 128 pixels of a phase (TMEM lanes), N = up to 128 input channels
// (TMEM columns), K = O per tap. A work unit is one band of phase rows of one
// image for one channel tile. g is read per pixel (g transposed to [B, Ho, Wo,
// O], bf16) and staged as a virtual image: row r, column v of the stage is g
// pixel (m0 + oh_min + r, ow_min + v), rows wv pixels wide (the widest phase
// plus the taps' spread), 128 bytes (64 channels) per pixel and slice. Output
// pixel (m0 + r, n) of a phase is virtual pixel r*wv + n, and tap (oh, ow)
// reads virtual pixel r*wv + n + shift, shift = (oh - oh_min)*wv + (ow -
// ow_min): a tap is a row offset of the A operand's start in shared memory.
// A band covers at most 256 virtual pixels: two 128-lane subtiles, the second
// starting 128 before the band's end (lanes the first one covered are not
// stored twice). Each chunk of O (kc 64-channel slices) is one copy of the
// band, each tap's weights of that chunk another (sign(w) as +-1 / 0 bf16 from
// bt_sign_transpose; bf16(scale_w) is applied to the fp32 accumulator).
//
// Warps: 0 copies (TMA), 1 issues the MMAs, 2..17 drain the accumulators:
// bf16 rounding, the mask from x, the grad_scale_a terms and the stores of
// gx (NCHW), each store instruction 32 consecutive pixels of one channel.
// Accumulators are double-buffered in TMEM so that a phase's epilogue runs
// under the next phase's MMAs.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda_bf16.h>

#include "bt_device.cuh"
#include "bt_internal.h"
#include "tc_ptx.cuh"

namespace bt {
namespace dgrad {

constexpr int kEpiWarps = 16;              // four per TMEM lane quarter, each its own 32-channel chunks
constexpr int kEpiGroups = kEpiWarps / 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;   // copies, MMAs, epilogue
constexpr int kMaxPhases = 16;             // strides up to 4
constexpr int kMaxTaps = 64;               // kernels up to 8 x 8
constexpr int kMaxW = 4;                   // weight ring slots
constexpr int kRow = 128;                  // bytes of a staged row: 64 bf16 channels
constexpr int kLanes = 128;                // pixels per subtile (MMA M)
constexpr int kBand = 256;                 // virtual pixels per band (two subtiles)
constexpr uint32_t kTmemCols = 512;
constexpr int kSmemMax = 227 * 1024;

struct DgArgs {
    int B, C, H, W, HW, Ho, Wo, s;
    int wv, R, hb, hn_max, nbands, nct, N, ncol;   // ncol: TMEM columns per subtile
    int kc, nchunks, nw, multi;                    // multi: one copy per chunk (else one per slice)
    int resident, ph_first, ph_last;               // resident: the band's chunks (<= 2) stay for all phases
    int oh_min, ow_min;
    int nph;
    int ph_rh[kMaxPhases], ph_rw[kMaxPhases], ph_hn[kMaxPhases], ph_wn[kMaxPhases];
    int ph_tap0[kMaxPhases], ph_ntap[kMaxPhases];
    int tap_shift[kMaxTaps], tap_w[kMaxTaps];
    int units;
    int ncg;                                       // 32-channel groups of x's codes per pixel
    uint32_t gslot, wslot, gbytes, wbytes, idesc;
    float alpha, bound, norm;
    const uint4 *codes;                            // x's mask and sign codes (code_kernel)
    __nv_bfloat16 *gx;
    float *sum;
    unsigned int *err;
    unsigned long long wait_ns;
};

__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap *m, int c0, int c1, int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_4d(uint32_t dst, const CUtensorMap *m, int c0, int c1, int c2, int c3,
                                       uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_5d(uint32_t dst, const CUtensorMap *m, int c0, int c1, int c2, int c3, int c4,
                                       uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
        : "memory");
}

// Per element of x, what the input gradient needs of it, as a nibble: bit 0
// set where the straight-through mask keeps the gradient (!(x < -bound || x >
// bound): |x| <= bound, or NaN), bit 1 where x > 0, bit 2 where x < 0. Laid
// out per pixel, 32 channels per 16 bytes: codes[(b*HW + pixel)*ncg + c/32],
// channel c at bits 4*(c%8) of word (c%32)/8; 0 past C. So the epilogue reads
// one 16-byte code per 32 channels of its pixel instead of 32 elements of x
// a plane apart.
// MMA and commit issued by the lanes with `issue` set (one lane): the issuing
// warp runs its loop converged, so the operand descriptors stay warp-uniform.
__device__ __forceinline__ void mma_bf16_if(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate,
                                            uint32_t issue) {
    asm volatile(
        "{\n"
        ".reg .pred p, q;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "setp.ne.b32 q, %5, 0;\n"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(issue)
        : "memory");
}
__device__ __forceinline__ void commit_if(uint32_t bar, uint32_t issue) {
    asm volatile(
        "{\n"
        ".reg .pred q;\n"
        "setp.ne.b32 q, %1, 0;\n"
        "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n"
        "}\n" ::"r"(bar), "r"(issue)
        : "memory");
}

template <typename XT> __device__ __forceinline__ float x_f32(const XT *p);
template <> __device__ __forceinline__ float x_f32<float>(const float *p) { return __ldg(p); }
template <> __device__ __forceinline__ float x_f32<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(__ldg(p));
}
constexpr int kCodeThreads = 256;
template <typename XT>
__global__ void __launch_bounds__(kCodeThreads) code_kernel(const XT *__restrict__ x, int64_t npix, int64_t hw, int C,
                                                            int ncg, float bound, uint4 *__restrict__ codes) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t pxl = static_cast<int64_t>(blockIdx.x) * kCodeThreads + threadIdx.x;   // b*HW + pixel
    if (pxl >= npix) return;
    const int cg = static_cast<int>(blockIdx.y);
    const int64_t b = pxl / hw, pix = pxl - b * hw;
    const XT *xp = x + (b * C + 32 * cg) * hw + pix;
    const int nc = C - 32 * cg < 32 ? C - 32 * cg : 32;
    float v[32];
    if (nc == 32) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = x_f32<XT>(xp + j * hw);
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = j < nc ? x_f32<XT>(xp + j * hw) : 0.0f;
    }
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const uint32_t nib = (fabsf(v[j]) > bound ? 0u : 1u) | (v[j] > 0.0f ? 2u : 0u) | (v[j] < 0.0f ? 4u : 0u);
        w[j / 8] |= (j < nc ? nib : 0u) << (4 * (j % 8));
    }
    codes[pxl * ncg + cg] = make_uint4(w[0], w[1], w[2], w[3]);
}

// One element of the input gradient from its fp32 accumulator and x's code
// nibble: y = bf16(acc * alpha) (one rounding), times 1 where the mask keeps
// it and 0 where not (a product, as the definition's); returns its bf16 bits
// and sets term = y_masked * sign(x) * norm, its grad_scale_a term (y_masked
// * sign(x) is exact, so one rounding of y_masked * (+-norm) is the same).
__device__ __forceinline__ uint32_t grad_elem(uint32_t acc, uint32_t nib, float alpha, float norm, float &term) {
    const float y = __uint_as_float(static_cast<uint32_t>(__bfloat16_as_ushort(
                        __float2bfloat16_rn(__fmul_rn(__uint_as_float(acc), alpha)))) << 16);
    const float ym = __fmul_rn(y, (nib & 1u) ? 1.0f : 0.0f);
    term = __fmul_rn(ym, (nib & 2u) ? norm : ((nib & 4u) ? -norm : 0.0f));
    return __float_as_uint(ym) >> 16;                          // ym is a bf16 value
}

// 2-byte store under a predicate (no branch around it).
__device__ __forceinline__ void st_b16_if(uint16_t *p, uint32_t v, bool pred) {
    asm volatile(
        "{\n"
        ".reg .pred q;\n"
        "setp.ne.b32 q, %2, 0;\n"
        "@q st.global.b16 [%0], %1;\n"
        "}\n" ::"l"(p), "h"(static_cast<uint16_t>(v)), "r"(static_cast<uint32_t>(pred))
        : "memory");
}

// Unit u -> image, band, channel tile; the band's first phase row, its
// virtual pixels and subtiles (the second subtile starts at nvb - 128).
struct Unit {
    int b, m0, nvb, nsub, c0;
};
__device__ __forceinline__ Unit unit_of(const DgArgs &a, int u) {
    Unit t;
    const int ct = u % a.nct;
    const int rest = u / a.nct;
    const int band = rest % a.nbands;
    t.b = rest / a.nbands;
    t.m0 = band * a.hb;
    const int rows = a.hn_max - t.m0 < a.hb ? a.hn_max - t.m0 : a.hb;
    t.nvb = rows * a.wv;
    t.nsub = t.nvb > kLanes ? 2 : 1;
    t.c0 = ct * a.N;
    return t;
}

__global__ void __launch_bounds__(kThreads, 1)
dgrad_kernel(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmW,
             const __grid_constant__ DgArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sG = base, sW = base + 2u * a.gslot;
    const uint32_t bars = sW + static_cast<uint32_t>(a.nw) * a.wslot;
    // gfull[2], gempty[2], wfull[kMaxW], wempty[kMaxW], tfull[2], tempty[2], drain
    auto gfull = [&](int i) { return bars + 8u * i; };
    auto gempty = [&](int i) { return bars + 8u * (2 + i); };
    auto wfull = [&](int i) { return bars + 8u * (4 + i); };
    auto wempty = [&](int i) { return bars + 8u * (4 + kMaxW + i); };
    auto tfull = [&](int i) { return bars + 8u * (4 + 2 * kMaxW + i); };
    auto tempty = [&](int i) { return bars + 8u * (6 + 2 * kMaxW + i); };
    const uint32_t drain = bars + 8u * (8 + 2 * kMaxW);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem_raw + (drain + 8u - raw));
    volatile uint32_t *abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(gfull(i), 1);
            tc::mbar_init(gempty(i), 1);
            tc::mbar_init(tfull(i), 1);
            tc::mbar_init(tempty(i), kEpiWarps);
        }
        for (int i = 0; i < kMaxW; ++i) {
            tc::mbar_init(wfull(i), 1);
            tc::mbar_init(wempty(i), 1);
        }
        tc::mbar_init(drain, 1);
        *abort_flag = 0u;
        tc::fence_mbar_init();
        tc::prefetch_map(&tmG);
        tc::prefetch_map(&tmW);
    }
    if (warp == 1) {
        tc::tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t buf_cols = 2u * static_cast<uint32_t>(a.ncol);

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- copies ----------------
            pdl_wait();                                   // g per pixel comes from the previous kernel
            int gs = 0, ws = 0;
            uint32_t gph = 0, wph = 0;
            uint32_t g_last[2] = {2u, 2u}, w_last[kMaxW] = {2u, 2u, 2u, 2u};   // phase of each slot's last copy
            bool ok = true;
            // chunk q of the band into slot gs: once per unit where the chunks stay
            // resident (slot q), else once per phase through the two-slot ring
            auto load_g = [&](const Unit &t, int q, int slot, uint32_t parity) {
                if (!tc::wait_fast(gempty(slot), parity ^ 1u, abort_flag, a.err, a.wait_ns)) return false;
                const uint32_t gdst = sG + static_cast<uint32_t>(slot) * a.gslot;
                tc::mbar_arrive_expect_tx(gfull(slot), a.gbytes);
                if (a.multi) {
                    tma_5d(gdst, &tmG, 0, a.ow_min, t.m0 + a.oh_min, q * a.kc, t.b, gfull(slot));
                } else {
                    const uint32_t slab = static_cast<uint32_t>(a.R * a.wv * kRow);
                    for (int j = 0; j < a.kc; ++j)
                        tma_4d(gdst + j * slab, &tmG, (q * a.kc + j) * 64, a.ow_min, t.m0 + a.oh_min, t.b, gfull(slot));
                }
                g_last[slot] = parity;
                return true;
            };
            for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
                const Unit t = unit_of(a, u);
                if (a.resident && a.ph_first >= 0) {
                    for (int q = 0; q < a.nchunks && ok; ++q) ok = load_g(t, q, q, gph);
                    gph ^= 1u;
                }
                for (int p = 0; p < a.nph && ok; ++p) {
                    const int nt = a.ph_ntap[p];
                    if (nt == 0) continue;
                    for (int q = 0; q < a.nchunks && ok; ++q) {
                        if (!a.resident) {
                            if (!load_g(t, q, gs, gph)) { ok = false; break; }
                            if (++gs == 2) { gs = 0; gph ^= 1u; }
                        }
                        for (int i = 0; i < nt; ++i) {
                            if (!tc::wait_fast(wempty(ws), wph ^ 1u, abort_flag, a.err, a.wait_ns)) { ok = false; break; }
                            const uint32_t wdst = sW + static_cast<uint32_t>(ws) * a.wslot;
                            const int tw = a.tap_w[a.ph_tap0[p] + i];
                            tc::mbar_arrive_expect_tx(wfull(ws), a.wbytes);
                            if (a.multi) {
                                tma_4d(wdst, &tmW, 0, t.c0, q * a.kc, tw, wfull(ws));
                            } else {
                                const uint32_t slab = static_cast<uint32_t>(a.N * kRow);
                                for (int j = 0; j < a.kc; ++j)
                                    tma_3d(wdst + j * slab, &tmW, (q * a.kc + j) * 64, tw, t.c0, wfull(ws));
                            }
                            w_last[ws] = wph;
                            if (++ws == a.nw) { ws = 0; wph ^= 1u; }
                        }
                    }
                }
            }
            if (!ok) {
                // every issued copy lands before the CTA can exit
                for (int i = 0; i < 2; ++i) {
                    if (g_last[i] < 2u) {
                        const unsigned long long t0 = globaltimer_ns();
                        while (!tc::mbar_try_wait(gfull(i), g_last[i]) && globaltimer_ns() - t0 < kWaitNs) {}
                    }
                }
                for (int i = 0; i < kMaxW; ++i) {
                    if (w_last[i] < 2u) {
                        const unsigned long long t0 = globaltimer_ns();
                        while (!tc::mbar_try_wait(wfull(i), w_last[i]) && globaltimer_ns() - t0 < kWaitNs) {}
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer (the whole warp, converged; lane 0 issues) ----------------
        const uint32_t issue = lane == 0 ? 1u : 0u;
        int gs = 0, ws = 0, local = 0;
        uint32_t gph = 0, wph = 0;
        bool ok = true;
        const uint32_t gslab = static_cast<uint32_t>(a.R * a.wv);   // rows of one slice of a staged chunk
        for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
            const Unit t = unit_of(a, u);
            const uint32_t st1 = t.nsub > 1 ? static_cast<uint32_t>(t.nvb - kLanes) : 0u;
            for (int p = 0; p < a.nph && ok; ++p) {
                const int nt = a.ph_ntap[p];
                if (nt == 0) continue;
                const int buf = local & 1;
                if (local >= 2) {
                    if (!tc::wait_fast(tempty(buf), static_cast<uint32_t>((local - 2) >> 1) & 1u, abort_flag,
                                          a.err, a.wait_ns)) { ok = false; break; }
                    tc::fence_after_sync();
                }
                const uint32_t d = tmem + static_cast<uint32_t>(buf) * buf_cols;
                const uint32_t d1 = d + static_cast<uint32_t>(a.ncol);
                for (int q = 0; q < a.nchunks && ok; ++q) {
                    const int slot = a.resident ? q : gs;
                    if (!a.resident || p == a.ph_first) {
                        if (!tc::wait_fast(gfull(slot), gph, abort_flag, a.err, a.wait_ns)) { ok = false; break; }
                        tc::fence_after_sync();
                    }
                    const uint32_t gA = sG + static_cast<uint32_t>(slot) * a.gslot;
                    for (int i = 0; i < nt; ++i) {
                        if (!tc::wait_fast(wfull(ws), wph, abort_flag, a.err, a.wait_ns)) { ok = false; break; }
                        tc::fence_after_sync();
                        const uint32_t wB = sW + static_cast<uint32_t>(ws) * a.wslot;
                        const uint32_t shift = static_cast<uint32_t>(a.tap_shift[a.ph_tap0[p] + i]);
                        const uint64_t a0 = tc::sw128_kmajor_desc(gA + shift * kRow);
                        const uint64_t a1 = tc::sw128_kmajor_desc(gA + (shift + st1) * kRow);
                        const uint64_t b0 = tc::sw128_kmajor_desc(wB);
                        const uint32_t first = (q | i) == 0 ? 1u : 0u;
                        for (int j = 0; j < a.kc; ++j) {
                            // descriptor start addresses count 16-byte units
                            const uint64_t aj = static_cast<uint64_t>(j) * gslab * (kRow >> 4);
                            const uint64_t bj = static_cast<uint64_t>(j) * static_cast<uint32_t>(a.N) * (kRow >> 4);
                            const uint32_t acc0 = (first && j == 0) ? 0u : 1u;
                            if (t.nsub > 1) {
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk) {
                                    const uint64_t bd = b0 + bj + 2 * kk;
                                    mma_bf16_if(d, a0 + aj + 2 * kk, bd, a.idesc, kk ? 1u : acc0, issue);
                                    mma_bf16_if(d1, a1 + aj + 2 * kk, bd, a.idesc, kk ? 1u : acc0, issue);
                                }
                            } else {
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    mma_bf16_if(d, a0 + aj + 2 * kk, b0 + bj + 2 * kk, a.idesc, kk ? 1u : acc0, issue);
                            }
                        }
                        commit_if(wempty(ws), issue);            // the weights' slot is free once these finish
                        if (++ws == a.nw) { ws = 0; wph ^= 1u; }
                    }
                    if (!ok) break;
                    if (!a.resident) {
                        commit_if(gempty(gs), issue);
                        if (++gs == 2) { gs = 0; gph ^= 1u; }
                    } else if (p == a.ph_last) {
                        commit_if(gempty(q), issue);             // the chunk's last phase: the slot is free
                    }
                }
                if (!ok) break;
                commit_if(tfull(buf), issue);
                ++local;
            }
            if (a.resident && a.ph_first >= 0) gph ^= 1u;
        }
        // every MMA issued finishes before the accumulators are freed
        commit_if(drain, issue);
        const unsigned long long t0 = globaltimer_ns();
        while (!tc::mbar_try_wait(drain, 0u) && globaltimer_ns() - t0 < kWaitNs) {}
        __syncwarp();
    } else {
        // ---------------- epilogue (warps 2..17) ----------------
        pdl_wait();
        const int quarter = warp & 3;                              // TMEM lanes this warp may read
        const int group = (warp - 2) >> 2;                         // its 32-channel chunks: kEpiGroups*j + group
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int li = quarter * 32 + lane;                        // this thread's lane in a subtile
        const int64_t HW = a.HW;
        const float alpha = a.alpha, norm = a.norm;
        uint16_t *const gx16 = reinterpret_cast<uint16_t *>(a.gx);
        const uint4 *const codes = a.codes;
        const int ncg = a.ncg;
        float tsum = 0.0f;
        int local = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
            const Unit t = unit_of(a, u);
            const int nc = a.C - t.c0 < a.N ? a.C - t.c0 : a.N;    // channels of this tile
            for (int p = 0; p < a.nph; ++p) {
                const bool has = a.ph_ntap[p] > 0;
                const int buf = local & 1;
                if (has) {
                    if (!tc::wait_fast(tfull(buf), static_cast<uint32_t>(local >> 1) & 1u, abort_flag, a.err,
                                          a.wait_ns)) { ok = false; break; }
                    tc::fence_after_sync();
                }
                const int rh = a.ph_rh[p], rw = a.ph_rw[p], hn = a.ph_hn[p], wn = a.ph_wn[p];
                for (int sub = 0; sub < t.nsub; ++sub) {
                    const int v = (sub == 0 ? 0 : t.nvb - kLanes) + li;
                    const int r = v / a.wv, n = v - r * a.wv, m = t.m0 + r;
                    const bool live = v < t.nvb && (sub == 0 || v >= kLanes) && n < wn && m < hn;
                    if (!__any_sync(0xFFFFFFFFu, live)) continue;
                    // lanes with no pixel read the tile's first pixel instead (loads need no
                    // predicate); only their stores and sum terms are dropped
                    const int64_t pix = live ? static_cast<int64_t>(a.s * m + rh) * a.W + (a.s * n + rw) : 0;
                    const int64_t off0 = (static_cast<int64_t>(t.b) * a.C + t.c0) * HW + pix;
                    const uint4 *cp = codes + (static_cast<int64_t>(t.b) * HW + pix) * ncg + t.c0 / 32;
                    const uint32_t tcol = tmem + lane_base + static_cast<uint32_t>(buf) * buf_cols +
                                          static_cast<uint32_t>(sub * a.ncol);
                    const uint32_t hw = static_cast<uint32_t>(HW);     // < 2^26: 32 planes in 32 bits
                    if (!has) {
                        // a phase no tap reaches: zeros
                        for (int c32 = 32 * group; c32 < nc; c32 += 32 * kEpiGroups) {
                            const int lim = nc - c32 < 32 ? nc - c32 : 32;
                            uint16_t *gp = gx16 + off0 + static_cast<int64_t>(c32) * HW;
                            if (live)
                                for (int rr = 0; rr < lim; ++rr) gp[rr * hw] = 0;
                        }
                        continue;
                    }
                    // codes past C are 0 and a lane with no pixel takes 0 codes, so its terms
                    // are zeros and only its stores need a predicate
                    for (int c32 = 32 * group; c32 < nc; c32 += 32 * kEpiGroups) {
                        const int lim = nc - c32 < 32 ? nc - c32 : 32;  // channels of this chunk (warp-uniform)
                        uint32_t acc[32];
                        tc::tmem_ld32(tcol + static_cast<uint32_t>(c32), acc);
                        const uint4 code = __ldg(cp + c32 / 32);
                        uint16_t *gp = gx16 + off0 + static_cast<int64_t>(c32) * HW;
                        const uint32_t cw[4] = {live ? code.x : 0u, live ? code.y : 0u, live ? code.z : 0u,
                                                live ? code.w : 0u};
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int rr = 0; rr < 32; ++rr) {
                            float term;
                            const uint32_t g16 = grad_elem(acc[rr], cw[rr / 8] >> (4 * (rr % 8)), alpha, norm, term);
                            tsum = __fadd_rn(tsum, term);
                            st_b16_if(gp + rr * hw, g16, live && rr < lim);
                        }
                    }
                }
                if (has) {
                    // this warp's reads of the buffer are complete
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(tempty(buf));
                    ++local;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tsum += __shfl_xor_sync(0xFFFFFFFFu, tsum, o);
        if (lane == 0) atomicAdd(a.sum, tsum);
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// Tiles, phases and taps of a layer; false where this kernel does not apply.
bool plan(int64_t B, int64_t C, int64_t H, int64_t W, int64_t O, int k, int s, int p, int d, DgArgs &a, int &smem) {
    if (B < 1 || O % 64 != 0 || s > 4 || k * k > kMaxTaps || C > int64_t(65535) * 32) return false;   // grid.y of the codes
    const int64_t Ho = (H + 2 * static_cast<int64_t>(p) - static_cast<int64_t>(d) * (k - 1) - 1) / s + 1;
    const int64_t Wo = (W + 2 * static_cast<int64_t>(p) - static_cast<int64_t>(d) * (k - 1) - 1) / s + 1;
    if (Ho < 1 || Wo < 1 || H * W >= (int64_t(1) << 26) || B * C * H * W > (int64_t(1) << 40)) return false;
    a = DgArgs{};
    a.B = static_cast<int>(B); a.C = static_cast<int>(C); a.H = static_cast<int>(H); a.W = static_cast<int>(W);
    a.HW = static_cast<int>(H * W); a.Ho = static_cast<int>(Ho); a.Wo = static_cast<int>(Wo); a.s = s;
    // phases and their taps; offsets (oh, ow) over every tap
    int oh_min = 0, oh_max = 0, ow_min = 0, ow_max = 0, ntaps = 0;
    int tap_oh[kMaxTaps], tap_ow[kMaxTaps];
    bool any = false;
    int nph = 0;
    for (int rh = 0; rh < s && rh < H; ++rh) {
        for (int rw = 0; rw < s && rw < W; ++rw) {
            a.ph_rh[nph] = rh;
            a.ph_rw[nph] = rw;
            a.ph_hn[nph] = static_cast<int>((H - rh + s - 1) / s);
            a.ph_wn[nph] = static_cast<int>((W - rw + s - 1) / s);
            a.ph_tap0[nph] = ntaps;
            for (int kh = 0; kh < k; ++kh) {
                const int th = rh + p - kh * d;
                if (((th % s) + s) % s != 0) continue;
                for (int kw = 0; kw < k; ++kw) {
                    const int tw = rw + p - kw * d;
                    if (((tw % s) + s) % s != 0) continue;
                    const int oh = floor_div(th, s), ow = floor_div(tw, s);
                    if (!any || oh < oh_min) oh_min = oh;
                    if (!any || oh > oh_max) oh_max = oh;
                    if (!any || ow < ow_min) ow_min = ow;
                    if (!any || ow > ow_max) ow_max = ow;
                    any = true;
                    tap_oh[ntaps] = oh;
                    tap_ow[ntaps] = ow;
                    a.tap_w[ntaps] = kh * k + kw;
                    ++ntaps;
                }
            }
            a.ph_ntap[nph] = ntaps - a.ph_tap0[nph];
            ++nph;
        }
    }
    a.nph = nph;
    a.hn_max = static_cast<int>((H + s - 1) / s);
    const int wn_max = static_cast<int>((W + s - 1) / s);
    a.wv = wn_max + (ow_max - ow_min);
    if (a.wv > kBand) return false;
    a.oh_min = oh_min;
    a.ow_min = ow_min;
    for (int i = 0; i < ntaps; ++i) a.tap_shift[i] = (tap_oh[i] - oh_min) * a.wv + (tap_ow[i] - ow_min);
    a.hb = a.hn_max < kBand / a.wv ? a.hn_max : kBand / a.wv;
    a.nbands = (a.hn_max + a.hb - 1) / a.hb;
    const int max_shift = (oh_max - oh_min) * a.wv + (ow_max - ow_min);
    const int nvb = a.hb * a.wv;
    a.R = ((nvb > kLanes ? nvb : kLanes) + max_shift + a.wv - 1) / a.wv;
    if (a.R > 256) return false;
    a.N = C >= 128 ? 128 : static_cast<int>((C + 15) / 16 * 16);
    a.ncol = (a.N + 31) / 32 * 32;
    a.nct = static_cast<int>((C + a.N - 1) / a.N);
    a.wslot = 0;
    // chunk of O per copy: the largest that leaves room for two chunks and two weight slots
    for (int kc = 4; kc >= 1; kc /= 2) {
        if (O % (64 * kc) != 0) continue;
        const uint32_t gslot = (static_cast<uint32_t>(a.R * a.wv * kRow * kc) + 1023u) & ~1023u;
        const uint32_t wslot = static_cast<uint32_t>(a.N * kRow * kc);
        const int fixed = 1024 + 2 * static_cast<int>(gslot) + 256;
        if (fixed + 2 * static_cast<int>(wslot) > kSmemMax) continue;
        int nw = (kSmemMax - fixed) / static_cast<int>(wslot);
        if (nw > kMaxW) nw = kMaxW;
        a.kc = kc;
        a.gslot = gslot;
        a.wslot = wslot;
        a.nw = nw;
        smem = fixed + nw * static_cast<int>(wslot);
        break;
    }
    if (a.wslot == 0) return false;
    a.nchunks = static_cast<int>(O / (64 * a.kc));
    a.resident = a.nchunks <= 2 ? 1 : 0;
    a.ph_first = -1;
    a.ph_last = -1;
    for (int i = 0; i < a.nph; ++i) {
        if (a.ph_ntap[i] == 0) continue;
        if (a.ph_first < 0) a.ph_first = i;
        a.ph_last = i;
    }
    a.gbytes = static_cast<uint32_t>(a.R * a.wv * kRow * a.kc);
    a.wbytes = static_cast<uint32_t>(a.N * kRow * a.kc);
    a.units = static_cast<int>(B) * a.nbands * a.nct;
    // BF16 x BF16 -> F32, K-major operands, M = 128, N
    a.idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((static_cast<uint32_t>(a.N) >> 3) << 17) | ((128u >> 4) << 24);
    return true;
}

// g per pixel [B, Ho, Wo, O] bf16 and the signs [k*k*C rows (c, kh, kw), ldw]
// as 128-byte swizzled boxes of 64 channels. One copy per chunk of kc slices
// (their strides out of order: the slice index strides 128 bytes), or, where
// the driver does not take that, one copy per slice.
bool encode(const DgArgs &a, int64_t O, int k, const uint16_t *g, const uint16_t *wst, int64_t ldw, bool multi,
            CUtensorMap *mg, CUtensorMap *mw) {
    auto fn = tensor_map_encoder();
    if (fn == nullptr) return false;
    const cuuint64_t e = 2;
    if (multi) {
        cuuint64_t gd[5] = {64, static_cast<cuuint64_t>(a.Wo), static_cast<cuuint64_t>(a.Ho),
                            static_cast<cuuint64_t>(O / 64), static_cast<cuuint64_t>(a.B)};
        cuuint64_t gs[4] = {O * e, static_cast<cuuint64_t>(a.Wo) * O * e, 128, static_cast<cuuint64_t>(a.Ho) * a.Wo * O * e};
        cuuint32_t gb[5] = {64, static_cast<cuuint32_t>(a.wv), static_cast<cuuint32_t>(a.R),
                            static_cast<cuuint32_t>(a.kc), 1};
        cuuint32_t es[5] = {1, 1, 1, 1, 1};
        if (fn(mg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<uint16_t *>(g), gd, gs, gb, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
        cuuint64_t wd[4] = {64, static_cast<cuuint64_t>(a.C), static_cast<cuuint64_t>(O / 64),
                            static_cast<cuuint64_t>(k * k)};
        cuuint64_t ws[3] = {static_cast<cuuint64_t>(k * k) * ldw * e, 128, ldw * e};
        cuuint32_t wb[4] = {64, static_cast<cuuint32_t>(a.N), static_cast<cuuint32_t>(a.kc), 1};
        return fn(mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t *>(wst), wd, ws, wb, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    cuuint64_t gd[4] = {static_cast<cuuint64_t>(O), static_cast<cuuint64_t>(a.Wo), static_cast<cuuint64_t>(a.Ho),
                        static_cast<cuuint64_t>(a.B)};
    cuuint64_t gs[3] = {O * e, static_cast<cuuint64_t>(a.Wo) * O * e, static_cast<cuuint64_t>(a.Ho) * a.Wo * O * e};
    cuuint32_t gb[4] = {64, static_cast<cuuint32_t>(a.wv), static_cast<cuuint32_t>(a.R), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (fn(mg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t *>(g), gd, gs, gb, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    cuuint64_t wd[3] = {static_cast<cuuint64_t>(O), static_cast<cuuint64_t>(k * k), static_cast<cuuint64_t>(a.C)};
    cuuint64_t ws[2] = {ldw * e, static_cast<cuuint64_t>(k * k) * ldw * e};
    cuuint32_t wb[3] = {64, 1, static_cast<cuuint32_t>(a.N)};
    return fn(mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(wst), wd, ws, wb, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_kernel(const CUtensorMap &mg, const CUtensorMap &mw, const DgArgs &a, int smem, cudaStream_t s) {
    auto kern = dgrad_kernel;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] { attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax); });
    if (attr_err != cudaSuccess) return attr_err;
    int grid = device_sm_count();
    if (grid > a.units) grid = a.units;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0] = pdl_attribute();
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, mg, mw, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename XT>
cudaError_t launch_codes(const XT *x, int64_t B, int64_t C, int64_t HW, float bound, uint4 *codes, cudaStream_t s) {
    const int ncg = static_cast<int>((C + 31) / 32);
    const int64_t npix = B * HW;
    return launch_pdl(code_kernel<XT>, dim3(static_cast<unsigned>((npix + kCodeThreads - 1) / kCodeThreads),
                                            static_cast<unsigned>(ncg)),
                      dim3(kCodeThreads), s, x, npix, HW, static_cast<int>(C), ncg, bound, codes);
}

// BT_CONV_DGRAD=gather in the environment turns this route off; =slices
// takes one copy per 64-channel slice.
int route_env() {
    const char *env = std::getenv("BT_CONV_DGRAD");
    if (env == nullptr) return 0;
    if (std::strcmp(env, "gather") == 0) return -1;
    if (std::strcmp(env, "slices") == 0) return 1;
    return 0;
}

}  // namespace dgrad

bool dgrad_implicit_applies(int64_t B, int64_t C, int64_t H, int64_t W, int64_t O, int k, int s, int p, int d) {
    if (dgrad::route_env() < 0) return false;
    dgrad::DgArgs a;
    int smem = 0;
    return dgrad::plan(B, C, H, W, O, k, s, p, d, a, smem);
}

size_t dgrad_codes_bytes(int64_t B, int64_t C, int64_t H, int64_t W) {
    return static_cast<size_t>(B * H * W * ((C + 31) / 32) * 16);
}

cudaError_t launch_dgrad_implicit(const uint16_t *g_nhwc, const uint16_t *wst, int64_t ldw, int64_t B, int64_t C,
                                  int64_t H, int64_t W, int64_t O, int k, int s, int p, int d, const void *x,
                                  bt_dtype x_dtype, float alpha, float bound, float norm, void *gx,
                                  float *sum, void *codes, unsigned int *err, cudaStream_t stream) {
    dgrad::DgArgs a;
    int smem = 0;
    if (!dgrad::plan(B, C, H, W, O, k, s, p, d, a, smem)) return cudaErrorNotSupported;
    if (reinterpret_cast<uintptr_t>(codes) % 16 != 0) return cudaErrorInvalidValue;
    a.alpha = alpha;
    a.bound = bound;
    a.norm = norm;
    a.ncg = static_cast<int>((C + 31) / 32);
    a.codes = static_cast<const uint4 *>(codes);
    a.gx = static_cast<__nv_bfloat16 *>(gx);
    a.sum = sum;
    a.err = err;
    a.wait_ns = wait_limit_ns();
    CUtensorMap mg, mw;
    bool multi = dgrad::route_env() != 1 && a.kc > 1;
    if (multi && !dgrad::encode(a, O, k, g_nhwc, wst, ldw, true, &mg, &mw)) multi = false;
    if (!multi && !dgrad::encode(a, O, k, g_nhwc, wst, ldw, false, &mg, &mw)) return cudaErrorInvalidValue;
    a.multi = multi ? 1 : 0;
    const cudaError_t e =
        x_dtype == BT_F32
            ? dgrad::launch_codes(static_cast<const float *>(x), B, C, H * W, bound, static_cast<uint4 *>(codes), stream)
            : dgrad::launch_codes(static_cast<const __nv_bfloat16 *>(x), B, C, H * W, bound, static_cast<uint4 *>(codes),
                                  stream);
    if (e != cudaSuccess) return e;
    return dgrad::launch_kernel(mg, mw, a, smem, stream);
}

}  // namespace bt
