// CUDA-core XOR + popcount contraction over BITS operands, for the linear
// layer (packed GEMM) and for the convolution (implicit im2col over
// channel-packed NHWC activations).
//
//   linear: dot[m,n] = K - 2 * sum_w popc(xp[m,w] ^ wp[n,w])
//   conv:   dot[b,o,i,j] = sum over taps t inside the image of
//                          (C - 2 * sum_w popc(xp[b,y_t,x_t,w] ^ wp[o,t,w]))
//                        = C * n_valid - 2 * acc
// Padding words are 0 in both operands and add nothing. A tap in the zero
// padding adds nothing either (the unfold + mm lowering of a convolution):
// its activation words are zero-filled and its popcounts masked out.
//
// A CTA owns a 128 x 128 output tile; 256 threads each hold 8 x 8
// accumulators. The reduction dimension is split into 4-word "slots" (a slot
// of the conv is 4 channel words of one tap); a pipeline stage holds two slots
// of A and B in shared memory, filled by cp.async with zero fill, three
// stages deep. Rows are padded to 12 words so that the 16-byte reads of eight
// consecutive rows hit eight different bank groups.
#include "bt_device.cuh"
#include "bt_internal.h"

namespace bt {
namespace {

constexpr int kBM = 128, kBN = 128, kThreads = 256;
constexpr int kLdw = 12;      // words per smem row (8 used)
constexpr int kStages = 3;

struct PopcArgs {
    const uint32_t *A;        // [M, Pw] (linear) or [B, H, W, Pw] (conv)
    const uint32_t *Bw;       // [N, Pw] (linear) or [O, k*k, Pw] (conv)
    int64_t M, N;
    int Pw;                   // words per packed row / per pixel
    int Kdot;                 // K (linear) or C (conv)
    int nslots;               // 4-word slots along the reduction
    float alpha;
    const float *scales;      // not null: alpha = fp32(scales[0] * scales[1]) read here
    void *out;
    // conv geometry
    int H, W, Ho, Wo, k, s, p, d;
};

template <bool CONV, int OUT>
__global__ void __launch_bounds__(kThreads) popc_kernel(const PopcArgs a) {
    __shared__ __align__(16) uint32_t As[kStages][kBM * kLdw];
    __shared__ __align__(16) uint32_t Bs[kStages][kBN * kLdw];
    __shared__ uint32_t Vs[kStages][2][kBM];   // conv: per-slot row masks

    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kBM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kBN;

    // This thread's load assignment: one 16-byte chunk (slot `ls`) of row `lr`
    // of A and of B per stage.
    const int lr = tid >> 1, ls = tid & 1;
    const int64_t am = m0 + lr, bn = n0 + lr;
    const bool a_row_ok = am < a.M, b_row_ok = bn < a.N;
    int ab = 0, ai = 0, aj = 0;
    if (CONV && a_row_ok) {
        const int64_t hw = static_cast<int64_t>(a.Ho) * a.Wo;
        ab = static_cast<int>(am / hw);
        const int pix = static_cast<int>(am - static_cast<int64_t>(ab) * hw);
        ai = pix / a.Wo;
        aj = pix - ai * a.Wo;
    }
    const int cpt = a.Pw >> 2;   // slots per tap (conv)
    const int nstages = (a.nslots + 1) >> 1;

    auto load_stage = [&](int buf, int g) {
        const int q = 2 * g + ls;
        const bool q_ok = q < a.nslots;
        // A
        const uint32_t *src = a.A;
        bool ok = a_row_ok && q_ok;
        if (CONV) {
            const int tap = q_ok ? q / cpt : 0;
            const int chunk = q_ok ? q - tap * cpt : 0;
            const int kh = tap / a.k, kw = tap - kh * a.k;
            const int y = ai * a.s - a.p + kh * a.d;
            const int x = aj * a.s - a.p + kw * a.d;
            ok = ok && y >= 0 && y < a.H && x >= 0 && x < a.W;
            if (ok) src = a.A + ((static_cast<int64_t>(ab) * a.H + y) * a.W + x) * a.Pw + chunk * 4;
            Vs[buf][ls][lr] = ok ? 0xFFFFFFFFu : 0u;
        } else if (ok) {
            src = a.A + am * a.Pw + q * 4;
        }
        cp_async_16(&As[buf][lr * kLdw + ls * 4], src, ok ? 16 : 0);
        // B
        const uint32_t *bsrc = a.Bw;
        const bool bok = b_row_ok && q_ok;
        if (bok) {
            if (CONV) {
                const int tap = q / cpt, chunk = q - tap * cpt;
                bsrc = a.Bw + (bn * (a.k * a.k) + tap) * a.Pw + chunk * 4;
            } else {
                bsrc = a.Bw + bn * a.Pw + q * 4;
            }
        }
        cp_async_16(&Bs[buf][lr * kLdw + ls * 4], bsrc, bok ? 16 : 0);
    };

    int acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0;

    // Rows of A and B this thread reads: the output index that is contiguous
    // in memory (n for a linear, the pixel for NCHW conv output) follows tx.
    int ra[8], rbw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        ra[i] = CONV ? tx + 16 * i : ty + 16 * i;
        rbw[i] = CONV ? ty + 16 * i : tx + 16 * i;
    }

#pragma unroll
    for (int st = 0; st < kStages - 1; ++st) {
        if (st < nstages) load_stage(st, st);
        cp_async_commit();
    }

    for (int g = 0; g < nstages; ++g) {
        cp_async_wait<kStages - 2>();
        __syncthreads();
        const int gn = g + kStages - 1;
        if (gn < nstages) load_stage(gn % kStages, gn);
        cp_async_commit();

        const int buf = g % kStages;
        const uint32_t *as = As[buf];
        const uint32_t *bs = Bs[buf];
#pragma unroll
        for (int sl = 0; sl < 2; ++sl) {
            uint4 av[8], bv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) av[i] = *reinterpret_cast<const uint4 *>(as + ra[i] * kLdw + sl * 4);
#pragma unroll
            for (int j = 0; j < 8; ++j) bv[j] = *reinterpret_cast<const uint4 *>(bs + rbw[j] * kLdw + sl * 4);
            uint32_t vm[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) vm[i] = CONV ? Vs[buf][sl][ra[i]] : 0xFFFFFFFFu;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int p = __popc(av[i].x ^ bv[j].x) + __popc(av[i].y ^ bv[j].y) +
                                  __popc(av[i].z ^ bv[j].z) + __popc(av[i].w ^ bv[j].w);
                    acc[i][j] += CONV ? static_cast<int>(static_cast<uint32_t>(p) & vm[i]) : p;
                }
            }
        }
    }
    cp_async_wait<0>();

    using OT = typename OutT<OUT>::type;
    OT *out = static_cast<OT *>(a.out);
    const float alpha = a.scales != nullptr ? alpha_from(a.scales) : a.alpha;
    if (!CONV) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t m = m0 + ra[i];
            if (m >= a.M) continue;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int64_t n = n0 + rbw[j];
                if (n < a.N) out[m * a.N + n] = OutT<OUT>::cvt(a.Kdot - 2 * acc[i][j], alpha);
            }
        }
    } else {
        const int64_t hw = static_cast<int64_t>(a.Ho) * a.Wo;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t m = m0 + ra[i];
            if (m >= a.M) continue;
            const int64_t b = m / hw;
            const int64_t pix = m - b * hw;
            const int oi = static_cast<int>(pix / a.Wo), oj = static_cast<int>(pix - (pix / a.Wo) * a.Wo);
            int nvh = 0, nvw = 0;
            for (int t = 0; t < a.k; ++t) {
                const int y = oi * a.s - a.p + t * a.d, x = oj * a.s - a.p + t * a.d;
                nvh += (y >= 0 && y < a.H);
                nvw += (x >= 0 && x < a.W);
            }
            const int base = a.Kdot * nvh * nvw;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int64_t o = n0 + rbw[j];
                if (o < a.N) out[(b * a.N + o) * hw + pix] = OutT<OUT>::cvt(base - 2 * acc[i][j], alpha);
            }
        }
    }
}

template <bool CONV>
cudaError_t launch(const PopcArgs &a, bt_dtype out_t, cudaStream_t s) {
    dim3 grid(static_cast<unsigned>((a.N + kBN - 1) / kBN), static_cast<unsigned>((a.M + kBM - 1) / kBM));
    switch (out_t) {
        case BT_F32: popc_kernel<CONV, BT_F32><<<grid, kThreads, 0, s>>>(a); break;
        case BT_BF16: popc_kernel<CONV, BT_BF16><<<grid, kThreads, 0, s>>>(a); break;
        case BT_F16: popc_kernel<CONV, BT_F16><<<grid, kThreads, 0, s>>>(a); break;
        default: popc_kernel<CONV, BT_I32><<<grid, kThreads, 0, s>>>(a); break;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_popc_linear(const uint32_t *xp, const uint32_t *wp, int64_t M, int64_t N, int64_t K,
                               float alpha, void *out, bt_dtype out_t, cudaStream_t s, const float *scales) {
    PopcArgs a{};
    a.A = xp; a.Bw = wp; a.M = M; a.N = N;
    a.Pw = static_cast<int>(row_bytes(K, BT_CODE_BITS) / 4);
    a.Kdot = static_cast<int>(K);
    a.nslots = a.Pw / 4;
    a.alpha = alpha; a.scales = scales; a.out = out;
    return launch<false>(a, out_t, s);
}

cudaError_t launch_popc_conv(const uint32_t *xp, const uint32_t *wp, const ConvGeom &g, float alpha,
                             void *out, bt_dtype out_t, cudaStream_t s, const float *scales) {
    PopcArgs a{};
    a.A = xp; a.Bw = wp;
    a.M = g.B * g.Ho * g.Wo; a.N = g.O;
    a.Pw = static_cast<int>(row_bytes(g.C, BT_CODE_BITS) / 4);
    a.Kdot = static_cast<int>(g.C);
    a.nslots = g.k * g.k * (a.Pw / 4);
    a.alpha = alpha; a.scales = scales; a.out = out;
    a.H = static_cast<int>(g.H); a.W = static_cast<int>(g.W);
    a.Ho = static_cast<int>(g.Ho); a.Wo = static_cast<int>(g.Wo);
    a.k = g.k; a.s = g.s; a.p = g.p; a.d = g.d;
    return launch<true>(a, out_t, s);
}

}  // namespace bt
