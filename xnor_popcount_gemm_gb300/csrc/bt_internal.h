// Host-side declarations shared by the translation units of libbt.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "bt.h"

namespace bt {

// Element and code helpers --------------------------------------------------
inline int dtype_bytes(bt_dtype t) {
    switch (t) {
        case BT_F32: case BT_I32: return 4;
        case BT_BF16: case BT_F16: return 2;
        default: return 0;
    }
}

// Bytes of one packed row: BITS rows round up to 16 bytes; E4M3 / E2M1 rows
// to 64 bytes, so that a row splits into whole 64- or 128-byte swizzle rows.
inline int64_t row_bytes(int64_t k, bt_code code) {
    switch (code) {
        case BT_CODE_BITS: return (((k + 31) / 32) * 4 + 15) / 16 * 16;
        case BT_CODE_E4M3: return (k + 63) / 64 * 64;
        case BT_CODE_E2M1: return ((k + 1) / 2 + 63) / 64 * 64;
        default: return -1;
    }
}

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Streaming multiprocessors of the current device (looked up once per device).
int device_sm_count();

// Device error word (a __device__ variable) as seen from the calling
// thread's current CUDA context. Returns nullptr on a CUDA error.
unsigned int *device_error_word();

// Limit of the tensor-core kernels' bounded waits, in ns (bt_set_wait_timeout;
// 2 s unless set).
unsigned long long wait_limit_ns();

// Unique id of the calling thread's current CUDA context (cuCtxGetId, never
// reused within the process). False when no context is current or the driver
// lacks the query.
bool current_context_id(unsigned long long *id);

// The device address of a __device__ variable belongs to one CUDA context:
// another context on the same device (a framework's own driver context, or
// the primary context again after cudaDeviceReset) holds its own copy of the
// module at another address. This cache keys the address by the current
// context's id. `lookup(void **)` runs cudaGetSymbolAddress in the translation
// unit that defines the variable (the host-side name of a __device__
// variable is a stand-in registered per translation unit) with the context
// current; it runs once per context, or on every call when no context id can
// be read.
struct SymbolAddressCache {
    static constexpr int kSlots = 16;
    std::mutex mu;
    unsigned long long ids[kSlots] = {};
    void *ptrs[kSlots] = {};
    int next = 0;

    template <typename Lookup> void *get(Lookup lookup, cudaError_t *err) {
        unsigned long long id = 0;
        bool keyed = current_context_id(&id);
        if (keyed) {
            std::lock_guard<std::mutex> lock(mu);
            for (int i = 0; i < kSlots; ++i)
                if (ptrs[i] != nullptr && ids[i] == id) return ptrs[i];
        }
        void *p = nullptr;
        *err = lookup(&p);
        if (*err != cudaSuccess) return nullptr;
        // the lookup may have made the device's primary context current
        if (!keyed) keyed = current_context_id(&id);
        if (keyed) {
            std::lock_guard<std::mutex> lock(mu);
            ids[next] = id;
            ptrs[next] = p;
            next = (next + 1) % kSlots;
        }
        return p;
    }
};

// Launchers (enqueue only; the caller has validated every argument) ---------
cudaError_t launch_pack_rows(const void *x, bt_dtype xt, int64_t R, int64_t K, const float *bias,
                             int64_t bias_len, bt_code code, void *out, cudaStream_t s);
cudaError_t launch_pack_nhwc(const void *x, bt_dtype xt, int64_t B, int64_t C, int64_t HW,
                             const float *bias, int64_t bias_len, bt_code code, void *out,
                             cudaStream_t s);

struct ConvGeom {
    int64_t B, C, H, W, O, Ho, Wo;
    int k, s, p, d;
};

// im2col rows: channel-packed pixels [B, H, W, row_bytes(C)] -> [B*Ho*Wo,
// k*k*row_bytes(C)], row (b, ho, wo) holding the packed pixel of every filter
// tap (kh, kw) in turn, zeros for a tap in the padding. Row bytes a multiple
// of 16.
cudaError_t launch_im2col_rows(const uint8_t *xp, const ConvGeom &g, int64_t rbc, uint8_t *rows,
                               cudaStream_t s);
// Bytes of that matrix.
inline int64_t im2col_bytes(const ConvGeom &g, int64_t rbc) { return g.B * g.Ho * g.Wo * g.k * g.k * rbc; }

// The contraction launchers scale by alpha, or, when `scales` is not null, by
// fp32(scales[0] * scales[1]) read on the device (two device floats: scale_a,
// scale_w), so that device-side scales need no host synchronisation.
cudaError_t launch_popc_linear(const uint32_t *xp, const uint32_t *wp, int64_t M, int64_t N,
                               int64_t K, float alpha, void *out, bt_dtype out_t, cudaStream_t s,
                               const float *scales = nullptr);
cudaError_t launch_popc_conv(const uint32_t *xp, const uint32_t *wp, const ConvGeom &g, float alpha,
                             void *out, bt_dtype out_t, cudaStream_t s, const float *scales = nullptr);

cudaError_t launch_tc_linear(const uint8_t *xp, const uint8_t *wp, bt_code code, int64_t M,
                             int64_t N, int64_t K, float alpha, void *out, bt_dtype out_t,
                             unsigned int *err, cudaStream_t s, const float *scales = nullptr);
// rows: the im2col rows of the packed input (launch_im2col_rows); output NCHW.
cudaError_t launch_tc_conv(const uint8_t *rows, const uint8_t *wp, bt_code code, const ConvGeom &g,
                           float alpha, void *out, bt_dtype out_t, unsigned int *err,
                           cudaStream_t s, const float *scales = nullptr);

// bf16 x bf16 contraction on the tensor cores (tcgen05 kind::f16, fp32
// accumulators), for the backward's products: a code value beside bt_code's.
constexpr int kCodeBF16 = 3;

// Straight-through mask applied by the bf16 contraction's epilogue: the
// output D [M, N] (bf16) is multiplied by middle = !(q < -1 || q > 1), q =
// x / scale_a rounded to x's dtype, x [M, N] of type x_t (BF16 or F32, row
// pitch N); and sum over D * sign(x) * norm is added to *sum (fp32 atomics).
struct TcMask {
    const void *x;
    bt_dtype x_t;
    float scale_a;
    float norm;
    float *sum;
};

// D[r, c] = alpha * sum_j A[r, j] * B[c, j] over bf16 rows: A [M, klen] with a
// row pitch of lda elements, B [N, klen] with pitch ldb; D row-major [M, N]
// (bf16 or f32; rounded to bf16 before any mask). klen, lda, ldb multiples
// of 8; with a mask, N a multiple of 8 and out 16-byte aligned.
cudaError_t launch_tc_bf16(const uint16_t *a, int64_t lda, const uint16_t *b, int64_t ldb, int64_t M, int64_t N,
                           int64_t klen, float alpha, void *out, bt_dtype out_t, const TcMask *mask,
                           unsigned int *err, cudaStream_t s);

// The same contraction split along K into `splits` equal parts (klen a
// multiple of 64 * splits), each part's fp32 partial sums (times alpha) in
// out [splits, M, N] (or, with nchw_hw > 0, each part laid out NCHW as a
// convolution's [N / nchw_hw images, M channels, nchw_hw pixels]); the caller
// adds them up.
cudaError_t launch_tc_bf16_splitk(const uint16_t *a, int64_t lda, const uint16_t *b, int64_t ldb, int64_t M,
                                  int64_t N, int64_t klen, int splits, float alpha, float *out, unsigned int *err,
                                  cudaStream_t s, int64_t nchw_hw = 0);

// out[c * ldo + r] = f(in[r * C + c]) as bf16 for r < R, c < C, and 0 for
// R <= r < ldo: f = torch.sign (sign = true; in of type in_t) or the value
// itself (sign = false; in bf16).
cudaError_t launch_transpose_bf16(const void *in, bt_dtype in_t, int64_t R, int64_t C, int64_t ldo, bool sign,
                                  uint16_t *out, cudaStream_t s);

// The same for `batch` matrices stored one after the other (in: R*C
// elements apart; out: C*ldo apart). batch <= 65535.
cudaError_t launch_transpose_bf16_batched(const void *in, bt_dtype in_t, int64_t R, int64_t C, int64_t ldo, bool sign,
                                          uint16_t *out, int batch, cudaStream_t s);

// Input gradient of the conv2d backward as one implicit GEMM (conv_dgrad.cu):
// g_nhwc = g per pixel [B, Ho, Wo, O] bf16, wst = the signs [C*k*k rows (c,
// kh, kw), ldw] bf16; writes gx [B, C, H, W] bf16 (bf16(alpha * sum), masked
// to 0 where x lies outside [-bound, bound]) and adds the grad_scale_a terms
// (times norm) to *sum. codes: dgrad_codes_bytes() of scratch (16-byte
// aligned) for x's mask and sign codes. applies: O a multiple of 64, stride
// <= 4, k*k <= 64, the layer's tiles fit (BT_CONV_DGRAD=gather turns the
// route off).
bool dgrad_implicit_applies(int64_t B, int64_t C, int64_t H, int64_t W, int64_t O, int k, int s, int p, int d);
size_t dgrad_codes_bytes(int64_t B, int64_t C, int64_t H, int64_t W);
cudaError_t launch_dgrad_implicit(const uint16_t *g_nhwc, const uint16_t *wst, int64_t ldw, int64_t B, int64_t C,
                                  int64_t H, int64_t W, int64_t O, int k, int s, int p, int d, const void *x,
                                  bt_dtype x_dtype, float alpha, float bound, float norm, void *gx,
                                  float *sum, void *codes, unsigned int *err, cudaStream_t stream);

// True when this build carries the tensor-core kernels.
bool tc_available();

// A launch shape of the linear layer's tensor-core contraction: CTA pairs
// (cta_group::2) or single CTAs, bn output columns per tile, d 128-byte K
// slices per pipeline stage, epi epilogue warps (4 or 8).
struct TcTileChoice {
    int pair, bn, d, epi;
};
// The shapes the measured selection times for an M x N x K linear contraction
// in `code` (E4M3 / E2M1) writing out_t: the cost model's own choice first,
// then the cheapest tile width by the model for every other (pair, d) with d
// of 1 to 4 K slices (the model itself picks among 1, 2 and 4), each
// with both epilogue warp counts, then narrower tiles (BN 192 down to 96) in
// the model's pairing and depth. Writes at most `max`; returns how many.
int tc_linear_candidates(int64_t M, int64_t N, int64_t K, bt_code code, bt_dtype out_t, TcTileChoice *out,
                         int max);
// The shape the calling thread's linear contractions take until cleared
// (nullptr): for timing one candidate.
void tc_linear_force(const TcTileChoice *c);
// Measured winners: the linear contractions of this device and (M, N, K,
// code, out_t) take `c` from now on. tc_linear_forget drops every entry.
void tc_linear_remember(int64_t M, int64_t N, int64_t K, bt_code code, bt_dtype out_t, const TcTileChoice &c);
void tc_linear_forget();
// True when a measured winner is kept for this device and key.
bool tc_linear_kept(int64_t M, int64_t N, int64_t K, bt_code code, bt_dtype out_t);

// The driver's cuTensorMapEncodeTiled (looked up once), or nullptr.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Fused shift + sign + pack + unfold for the tensor-core convolution: NCHW x
// straight to the im2col rows launch_im2col_rows would build from the packed
// pixels (codes E4M3 / E2M1). The staged kernel needs x's channel planes
// 16-byte aligned and a band of input rows that fits shared memory; otherwise
// a direct kernel runs when direct_ok, else cudaErrorNotSupported is returned
// (the caller packs to NHWC and unfolds in two kernels).
cudaError_t launch_pack_im2col(const void *x, bt_dtype xt, const ConvGeom &g, const float *bias, int64_t bias_len,
                               bt_code code, uint8_t *rows, bool direct_ok, cudaStream_t s);
// Whether the convolution builds its im2col rows in one pass from x (for a
// 16-byte aligned x of type xt): the staged plan exists and pays.
bool unfold_single_pass(const ConvGeom &g, bt_dtype xt, bt_code code);

// Implicit-im2col tensor-core convolution straight from channel-packed NHWC
// pixels xp [B, H, W, row_bytes(C)] (codes E4M3 / E2M1), NCHW output. Whether
// its plan applies to a geometry does not depend on O (g.O is ignored);
// BT_CONV_IMPLICIT=0 in the environment turns it off (the explicit unfold
// then runs). The launch returns cudaErrorNotSupported where the plan does
// not apply.
bool conv_implicit_applies(const ConvGeom &g, bt_code code);
// after_own_pack: the kernel launched just before on the stream is the
// library's pack of x (it writes the pixels only), so the weights may be read
// before the wait on that kernel.
cudaError_t launch_tc_conv_implicit(const uint8_t *xp, const uint8_t *wp, bt_code code, const ConvGeom &g, float alpha,
                                    void *out, bt_dtype out_t, unsigned int *err, cudaStream_t s,
                                    const float *scales = nullptr, bool after_own_pack = false);
// The same convolution reading x itself (NCHW floats of type x_dtype, shifted
// by bias (bias_len 1 or C; 0: none) and signed by its own packing warps): one
// kernel, no workspace. It applies where the implicit plan does, every
// channel plane (H * W values) is a multiple of 16 bytes and BT_CONV_FUSED=1
// is set in the environment (otherwise the pack kernel runs first).
bool conv_fused_applies(const ConvGeom &g, bt_code code, bt_dtype x_dtype);
cudaError_t launch_tc_conv_fused(const void *x, bt_dtype x_dtype, const float *bias, int64_t bias_len,
                                 const uint8_t *wp, bt_code code, const ConvGeom &g, float alpha, void *out,
                                 bt_dtype out_t, unsigned int *err, cudaStream_t s, const float *scales = nullptr);

// A launch plan of the implicit-im2col convolution, for the measured
// selection: CTA pairs or single CTAs, weights resident ('R') or streamed
// ('S'), 1 or 2 pixel stages, (fused = 1) the convolution packing x itself
// instead of the NHWC pack kernel running first, and (split > 1) each image
// cut into that many times the planner's bands (more, narrower tiles).
struct ConvChoice {
    int pair, plan, bst, fused, split;
};
// The plans the measured selection times for this geometry, code, input and
// output dtype: the planner's own first, then every other (pair, plan,
// stages) that fits, each also with 2 and 4 times the bands where that
// changes the tiling, then each of them packing x itself where that route
// applies (float x). Writes at most `max`; returns how many (0 where the
// implicit plan does not apply).
int conv_candidates(const ConvGeom &g, bt_code code, bt_dtype x_dtype, bt_dtype out_t, ConvChoice *out, int max);
// The plan the calling thread's convolutions take until cleared (nullptr);
// the environment's BT_CONV_PAIR / BT_CONV_PLAN / BT_CONV_FUSED come first.
void conv_force(const ConvChoice *c);
const ConvChoice *conv_forced();
// Measured winners per device, geometry (g.O included), code and output
// dtype; conv_kept_fused answers for any O and output dtype (the most
// recent entry of the geometry and code).
void conv_remember(const ConvGeom &g, bt_code code, bt_dtype out_t, const ConvChoice &c);
bool conv_lookup(const ConvGeom &g, bt_code code, bt_dtype out_t, ConvChoice &c);
bool conv_kept_fused(const ConvGeom &g, bt_code code, bool &fused);
void conv_forget();
// The tiling a convolution launch would take (host only, no CUDA call): sms
// SMs, pair -1 (the planner's choice), 0 or 1, split >= 1 times the bands.
// False where the implicit plan does not apply.
bool conv_plan_query(const ConvGeom &g, bt_code code, int out_elem, int sms, int pair, int split,
                     bt_conv_plan_info &info);

// First-call activation scale (BinaryConv2dCutlass.set_activation): the sum
// of |x| accumulates in a double per CUDA context (zero it before use; calls
// that overlap on one GPU share it); launch_abs_sum adds the sum of |x| of n
// elements to it in a separate pass; launch_scale_finish turns it into
// (factor * mean) rounded to x's dtype, then to scale_dtype, written to
// scale_out (one float).
double *fused_abs_sum_accumulator(cudaError_t *err);
cudaError_t launch_abs_sum(const void *x, bt_dtype x_dtype, int64_t n, double *acc, cudaStream_t s);
cudaError_t launch_scale_finish(const double *acc, int64_t n, float factor, bt_dtype x_dtype, bt_dtype scale_dtype,
                                float *scale_out, cudaStream_t s);

// The activation packs with the sum of |x| of every element they read added to
// *abs_sum (compensated fp32 per thread, double across warps): rows (the flat
// kernel) and channel-packed pixels (the warp-level kernel). They return
// cudaErrorNotSupported where those kernels do not apply; the caller then
// packs as usual and sums in a separate pass.
cudaError_t launch_pack_rows_sum(const void *x, bt_dtype xt, int64_t R, int64_t K, const float *bias,
                                 int64_t bias_len, bt_code code, void *out, double *abs_sum, cudaStream_t s);
cudaError_t launch_pack_nhwc_sum(const void *x, bt_dtype xt, int64_t B, int64_t C, int64_t HW, const float *bias,
                                 int64_t bias_len, bt_code code, void *out, double *abs_sum, cudaStream_t s);

// Launch attribute list allowing programmatic dependent launch (the kernel
// overlaps its prologue with the previous kernel in the stream).
inline cudaLaunchAttribute pdl_attribute() {
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    return a;
}

// Round a float to the nearest bf16 value (ties to even), as a float; inf and
// NaN unchanged.
inline float bf16_round_host(float v) {
    uint32_t u;
    __builtin_memcpy(&u, &v, 4);
    if ((u & 0x7F800000u) == 0x7F800000u) return v;
    u = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
    float r;
    __builtin_memcpy(&r, &u, 4);
    return r;
}

inline size_t round_up256(size_t v) { return (v + 255) / 256 * 256; }

// Launch `kern` on `s` with programmatic dependent launch allowed (and
// `smem` bytes of dynamic shared memory).
template <typename K, typename... Args>
cudaError_t launch_pdl_smem(K kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute pdl = pdl_attribute();
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = &pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename K, typename... Args>
cudaError_t launch_pdl(K kern, dim3 grid, dim3 block, cudaStream_t s, Args... args) {
    return launch_pdl_smem(kern, grid, block, 0, s, args...);
}

// Largest K (elements) for which the tensor-core kernels are used: a bound on
// the magnitude of the fp32 partial sums they accumulate.
constexpr int64_t kTcMaxK = 16384;

}  // namespace bt
