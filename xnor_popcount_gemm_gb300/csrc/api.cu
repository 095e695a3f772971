// The C ABI of libbt (declared in include/bt.h): argument validation, the
// pack -> contract dispatch, the "ADAPTIVE" planner and the device error word.
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <map>
#include <mutex>

#include "bt_device.cuh"
#include "bt_internal.h"

namespace bt {

__device__ unsigned int g_error_word;

int device_sm_count() {
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

namespace {
std::atomic<unsigned long long> g_wait_limit_ns{kWaitNs};
}  // namespace

unsigned long long wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

bool current_context_id(unsigned long long *id) {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (get_current == nullptr || get_id == nullptr) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

unsigned int *device_error_word() {
    static SymbolAddressCache cache;
    cudaError_t err = cudaSuccess;
    return static_cast<unsigned int *>(
        cache.get([](void **p) { return cudaGetSymbolAddress(p, g_error_word); }, &err));
}

namespace {

bool valid_code(int c) { return c == BT_CODE_BITS || c == BT_CODE_E4M3 || c == BT_CODE_E2M1; }
bool float_in(int t) { return t == BT_F32 || t == BT_BF16 || t == BT_F16; }
bool valid_out(int t) { return t == BT_F32 || t == BT_BF16 || t == BT_F16 || t == BT_I32; }
bool valid_scale(float v) { return std::isfinite(v) && v > 0.0f; }

// Timed calls per candidate when a call with BT_ALGO_TUNE tunes its size.
constexpr int kAutoTuneReps = 3;

// True while `s` is being captured into a graph (or when the query fails).
bool stream_capturing(cudaStream_t s) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return true;
    return cap != cudaStreamCaptureStatusNone;
}

bt_algo algo_for_code(bt_code c) {
    switch (c) {
        case BT_CODE_BITS: return BT_ALGO_POPC;
        case BT_CODE_E4M3: return BT_ALGO_TC_E4M3;
        default: return BT_ALGO_TC_E2M1;
    }
}

// alpha = fp32(scale_a * scale_w): the product of two floats is exact in
// double; one rounding to float.
float alpha_of(float sa, float sw) {
    return static_cast<float>(static_cast<double>(sa) * static_cast<double>(sw));
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bt_status from_cuda(cudaError_t e) { return e == cudaSuccess ? BT_OK : BT_ERR_CUDA; }

int64_t conv_out(int64_t h, int64_t k, int64_t s, int64_t p, int64_t d) {
    const int64_t num = h + 2 * p - d * (k - 1) - 1;
    return num < 0 ? 0 : num / s + 1;
}

// Largest reduction length whose dot fits exactly in an fp32 (|dot| <= 2^24).
constexpr int64_t kMaxK = int64_t(1) << 24;

}  // namespace
}  // namespace bt

using namespace bt;

extern "C" {

int bt_version(void) { return 100; }

const char *bt_status_string(bt_status s) {
    switch (s) {
        case BT_OK: return "BT_OK";
        case BT_ERR_INVALID_ARG: return "BT_ERR_INVALID_ARG: invalid argument";
        case BT_ERR_UNSUPPORTED: return "BT_ERR_UNSUPPORTED: unsupported combination";
        case BT_ERR_ALIGNMENT: return "BT_ERR_ALIGNMENT: pointer not aligned (16 B; workspace 256 B)";
        case BT_ERR_WORKSPACE: return "BT_ERR_WORKSPACE: workspace missing or too small";
        case BT_ERR_CUDA: return "BT_ERR_CUDA: CUDA error";
        case BT_ERR_TIMEOUT: return "BT_ERR_TIMEOUT: a kernel's bounded wait ran out";
        default: return "unknown bt_status";
    }
}

int64_t bt_packed_row_bytes(int64_t k, bt_code code) {
    if (k < 0 || !valid_code(code)) return -1;
    return row_bytes(k, code);
}

bt_status bt_pack_sign(const void *x, bt_dtype x_dtype, bt_layout layout, int64_t d0, int64_t d1,
                       int64_t d2, int64_t d3, const float *bias, int64_t bias_len, bt_code code,
                       void *out, bt_stream stream) {
    if (!valid_code(code) || !float_in(x_dtype)) return BT_ERR_INVALID_ARG;
    if (layout != BT_LAYOUT_ROWS && layout != BT_LAYOUT_NCHW_TO_NHWC) return BT_ERR_INVALID_ARG;
    if (d0 < 0 || d1 < 1) return BT_ERR_INVALID_ARG;
    if (layout == BT_LAYOUT_NCHW_TO_NHWC && (d2 < 1 || d3 < 1)) return BT_ERR_INVALID_ARG;
    if (!(bias_len == 0 || bias_len == 1 || bias_len == d1)) return BT_ERR_INVALID_ARG;
    if (bias_len > 0 && bias == nullptr) return BT_ERR_INVALID_ARG;
    if (d1 > (int64_t(1) << 30) || (layout == BT_LAYOUT_NCHW_TO_NHWC && (d2 * d3 > (int64_t(1) << 30) ||
                                                                        d0 > (int64_t(1) << 30))))
        return BT_ERR_UNSUPPORTED;
    if (d0 == 0) return BT_OK;
    if (x == nullptr || out == nullptr) return BT_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(out, 16) || (bias && !aligned(bias, 4))) return BT_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (layout == BT_LAYOUT_ROWS)
        return from_cuda(launch_pack_rows(x, x_dtype, d0, d1, bias, bias_len, code, out, s));
    return from_cuda(launch_pack_nhwc(x, x_dtype, d0, d1, d2 * d3, bias, bias_len, code, out, s));
}

size_t bt_binary_linear_workspace(int64_t M, int64_t K, bt_dtype x_dtype, bt_code code) {
    if (M < 0 || K < 1 || !valid_code(code) || x_dtype == BT_PACKED) return 0;
    return round_up(static_cast<size_t>(M) * static_cast<size_t>(row_bytes(K, code)), 256);
}

namespace {
// The forward with host scales (scales == nullptr) or device scales.
bt_status linear_impl(const void *x, bt_dtype x_dtype, const void *weight, bt_code w_code, int64_t M, int64_t N,
                      int64_t K, float scale_a, float scale_w, const float *scales, const float *bias_a,
                      int64_t bias_len, void *out, bt_dtype out_dtype, bt_algo algo, void *workspace,
                      size_t workspace_bytes, bt_stream stream) {
    if (!valid_code(w_code) || !valid_out(out_dtype)) return BT_ERR_INVALID_ARG;
    if (!(float_in(x_dtype) || x_dtype == BT_PACKED)) return BT_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 1) return BT_ERR_INVALID_ARG;
    if (scales == nullptr && (!valid_scale(scale_a) || !valid_scale(scale_w))) return BT_ERR_INVALID_ARG;
    if (!(bias_len == 0 || bias_len == 1 || bias_len == K)) return BT_ERR_INVALID_ARG;
    if (bias_len > 0 && bias_a == nullptr && x_dtype != BT_PACKED) return BT_ERR_INVALID_ARG;
    if (algo != BT_ALGO_AUTO && algo != algo_for_code(w_code)) {
        if (algo < BT_ALGO_AUTO || algo > BT_ALGO_TC_E2M1) return BT_ERR_INVALID_ARG;
        return BT_ERR_UNSUPPORTED;
    }
    if (K > kMaxK) return BT_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return BT_OK;
    if (x == nullptr || weight == nullptr || out == nullptr) return BT_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(weight, 16) || !aligned(out, 16)) return BT_ERR_ALIGNMENT;
    if (scales != nullptr && !aligned(scales, 8)) return BT_ERR_ALIGNMENT;
    if (M > int64_t(65535) * 128) return BT_ERR_UNSUPPORTED;              // at most 65535 row tiles of 128
    const bt_algo run = algo_for_code(w_code);
    if (run != BT_ALGO_POPC && K > kTcMaxK) return BT_ERR_UNSUPPORTED;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const void *xp = x;
    if (x_dtype != BT_PACKED) {
        const size_t need = bt_binary_linear_workspace(M, K, x_dtype, w_code);
        if (workspace == nullptr || workspace_bytes < need) return BT_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return BT_ERR_ALIGNMENT;
        cudaError_t e = launch_pack_rows(x, x_dtype, M, K, bias_a, bias_len, w_code, workspace, s);
        if (e != cudaSuccess) return BT_ERR_CUDA;
        xp = workspace;
    }
    const float alpha = alpha_of(scale_a, scale_w);
    if (run == BT_ALGO_POPC)
        return from_cuda(launch_popc_linear(static_cast<const uint32_t *>(xp),
                                            static_cast<const uint32_t *>(weight), M, N, K, alpha, out,
                                            out_dtype, s, scales));
    unsigned int *err = device_error_word();
    if (err == nullptr) return BT_ERR_CUDA;
    return from_cuda(launch_tc_linear(static_cast<const uint8_t *>(xp), static_cast<const uint8_t *>(weight),
                                      w_code, M, N, K, alpha, out, out_dtype, err, s, scales));
}
}  // namespace

bt_status bt_binary_linear(const void *x, bt_dtype x_dtype, const void *weight, bt_code w_code,
                           int64_t M, int64_t N, int64_t K, float scale_a, float scale_w,
                           const float *bias_a, int64_t bias_len, void *out, bt_dtype out_dtype,
                           bt_algo algo, void *workspace, size_t workspace_bytes, bt_stream stream) {
    if (algo == BT_ALGO_TUNE) {
        algo = BT_ALGO_AUTO;
        // a size with launch shapes to choose from and none kept yet: tune it
        // (the last timed call leaves this call's result in out)
        if ((w_code == BT_CODE_E4M3 || w_code == BT_CODE_E2M1) && M >= 1 && N >= 1 && K >= 1 && K <= kTcMaxK &&
            valid_out(out_dtype) && !tc_linear_kept(M, N, K, w_code, out_dtype) &&
            !stream_capturing(reinterpret_cast<cudaStream_t>(stream))) {
            bt_tune_result r;
            return bt_tune_linear(x, x_dtype, weight, w_code, M, N, K, scale_a, scale_w, bias_a, bias_len, out,
                                  out_dtype, workspace, workspace_bytes, kAutoTuneReps, stream, &r);
        }
    }
    return linear_impl(x, x_dtype, weight, w_code, M, N, K, scale_a, scale_w, nullptr, bias_a, bias_len, out,
                       out_dtype, algo, workspace, workspace_bytes, stream);
}

bt_status bt_binary_linear_dscale(const void *x, bt_dtype x_dtype, const void *weight, bt_code w_code, int64_t M,
                                  int64_t N, int64_t K, const float *scales, const float *bias_a, int64_t bias_len,
                                  void *out, bt_dtype out_dtype, bt_algo algo, void *workspace,
                                  size_t workspace_bytes, bt_stream stream) {
    if (scales == nullptr) return BT_ERR_INVALID_ARG;
    return linear_impl(x, x_dtype, weight, w_code, M, N, K, 1.0f, 1.0f, scales, bias_a, bias_len, out, out_dtype,
                       algo, workspace, workspace_bytes, stream);
}

bt_status bt_binary_linear_dscale_init(const void *x, bt_dtype x_dtype, const void *weight, bt_code w_code,
                                       int64_t M, int64_t N, int64_t K, float *scales, float factor,
                                       bt_dtype scale_dtype, const float *bias_a, int64_t bias_len, void *out,
                                       bt_dtype out_dtype, bt_algo algo, void *workspace, size_t workspace_bytes,
                                       bt_stream stream) {
    if (scales == nullptr || !float_in(x_dtype) || !float_in(scale_dtype)) return BT_ERR_INVALID_ARG;
    if (!(std::isfinite(factor) && factor > 0.0f)) return BT_ERR_INVALID_ARG;
    if (!valid_code(w_code) || !valid_out(out_dtype) || M < 0 || N < 0 || K < 1) return BT_ERR_INVALID_ARG;
    if (!(bias_len == 0 || bias_len == 1 || bias_len == K) || (bias_len > 0 && bias_a == nullptr))
        return BT_ERR_INVALID_ARG;
    if (K > kMaxK) return BT_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return BT_OK;
    if (x == nullptr || weight == nullptr || out == nullptr) return BT_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(weight, 16) || !aligned(out, 16) || !aligned(scales, 8)) return BT_ERR_ALIGNMENT;
    const size_t need = bt_binary_linear_workspace(M, K, x_dtype, w_code);
    if (workspace == nullptr || workspace_bytes < need) return BT_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return BT_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err = cudaSuccess;
    double *acc = fused_abs_sum_accumulator(&err);
    if (acc == nullptr || cudaMemsetAsync(acc, 0, sizeof(double), s) != cudaSuccess) return BT_ERR_CUDA;
    // pack x and sum |x| in the same pass (or, where the fused pack does not
    // apply, pack and sum in two)
    cudaError_t e = launch_pack_rows_sum(x, x_dtype, M, K, bias_a, bias_len, w_code, workspace, acc, s);
    if (e == cudaErrorNotSupported) {
        e = launch_pack_rows(x, x_dtype, M, K, bias_a, bias_len, w_code, workspace, s);
        if (e == cudaSuccess) e = launch_abs_sum(x, x_dtype, M * K, acc, s);
    }
    if (e != cudaSuccess) return BT_ERR_CUDA;
    if (launch_scale_finish(acc, M * K, factor, x_dtype, scale_dtype, scales, s) != cudaSuccess) return BT_ERR_CUDA;
    return linear_impl(workspace, BT_PACKED, weight, w_code, M, N, K, 1.0f, 1.0f, scales, nullptr, 0, out, out_dtype,
                       algo, nullptr, 0, stream);
}

size_t bt_binary_conv2d_workspace(int64_t B, int64_t C, int64_t H, int64_t W, int kernel_size, int stride,
                                  int padding, int dilation, bt_dtype x_dtype, bt_code code) {
    if (B < 0 || C < 1 || H < 1 || W < 1 || !valid_code(code) || x_dtype == BT_PACKED_IM2COL) return 0;
    if (kernel_size < 1 || stride < 1 || padding < 0 || dilation < 1) return 0;
    if (B > (int64_t(1) << 30) || C > kMaxK || H > (1 << 20) || W > (1 << 20) || kernel_size > 64 ||
        padding > (1 << 20) || stride > (1 << 20) || dilation > (1 << 10))
        return 0;
    const int64_t rbc = row_bytes(C, code);
    const double approx = static_cast<double>(B) * H * W * rbc +
                          static_cast<double>(B) * H * W * kernel_size * kernel_size * rbc;
    if (approx > 4.0e18) return 0;
    size_t n = 0;
    if (x_dtype != BT_PACKED) n += round_up(static_cast<size_t>(B * H * W * rbc), 256);   // packed NHWC pixels
    if (code != BT_CODE_BITS) {
        ConvGeom g{B, C, H, W, 0, 0, 0, kernel_size, stride, padding, dilation};
        g.Ho = conv_out(H, kernel_size, stride, padding, dilation);
        g.Wo = conv_out(W, kernel_size, stride, padding, dilation);
        // the implicit-im2col contraction reads the packed pixels as they are;
        // otherwise the im2col rows follow them
        if (g.Ho >= 1 && g.Wo >= 1 && !conv_implicit_applies(g, code))
            n += round_up(static_cast<size_t>(im2col_bytes(g, rbc)), 256);
    }
    return n;
}

namespace {
bt_status conv_impl(const void *x, bt_dtype x_dtype, const void *weight, bt_code w_code, int64_t B, int64_t C,
                    int64_t H, int64_t W, int64_t O, int kernel_size, int stride, int padding, int dilation,
                    float scale_a, float scale_w, const float *scales, const float *bias_a, int64_t bias_len,
                    void *out, bt_dtype out_dtype, bt_algo algo, void *workspace, size_t workspace_bytes,
                    bt_stream stream) {
    if (!valid_code(w_code) || !valid_out(out_dtype)) return BT_ERR_INVALID_ARG;
    if (!(float_in(x_dtype) || x_dtype == BT_PACKED || x_dtype == BT_PACKED_IM2COL)) return BT_ERR_INVALID_ARG;
    if (x_dtype == BT_PACKED_IM2COL && w_code == BT_CODE_BITS) return BT_ERR_INVALID_ARG;
    if (B < 0 || C < 1 || H < 1 || W < 1 || O < 0) return BT_ERR_INVALID_ARG;
    if (kernel_size < 1 || stride < 1 || padding < 0 || dilation < 1) return BT_ERR_INVALID_ARG;
    if (scales == nullptr && (!valid_scale(scale_a) || !valid_scale(scale_w))) return BT_ERR_INVALID_ARG;
    if (!(bias_len == 0 || bias_len == 1 || bias_len == C)) return BT_ERR_INVALID_ARG;
    if (bias_len > 0 && bias_a == nullptr && float_in(x_dtype)) return BT_ERR_INVALID_ARG;
    if (algo != BT_ALGO_AUTO && algo != algo_for_code(w_code)) {
        if (algo < BT_ALGO_AUTO || algo > BT_ALGO_TC_E2M1) return BT_ERR_INVALID_ARG;
        return BT_ERR_UNSUPPORTED;
    }
    ConvGeom g{B, C, H, W, O, 0, 0, kernel_size, stride, padding, dilation};
    g.Ho = conv_out(H, kernel_size, stride, padding, dilation);
    g.Wo = conv_out(W, kernel_size, stride, padding, dilation);
    if (g.Ho < 1 || g.Wo < 1) return BT_ERR_INVALID_ARG;
    const int64_t kk = static_cast<int64_t>(kernel_size) * kernel_size;
    if (C > kMaxK || kernel_size > 64 || C * kk > kMaxK || H > (1 << 20) || W > (1 << 20) || padding > (1 << 20) ||
        stride > (1 << 20) || dilation > (1 << 10))
        return BT_ERR_UNSUPPORTED;
    if (B == 0 || O == 0) return BT_OK;
    if (x == nullptr || weight == nullptr || out == nullptr) return BT_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(weight, 16) || !aligned(out, 16)) return BT_ERR_ALIGNMENT;
    if (scales != nullptr && !aligned(scales, 8)) return BT_ERR_ALIGNMENT;
    // at most 65535 pixel tiles of 128 (each factor bounded first, so the product stays in range)
    if (B > int64_t(65535) * 128 || g.Ho * g.Wo > int64_t(65535) * 128) return BT_ERR_UNSUPPORTED;
    const int64_t M = B * g.Ho * g.Wo;
    if (M > int64_t(65535) * 128) return BT_ERR_UNSUPPORTED;
    const bt_algo run = algo_for_code(w_code);
    if (run != BT_ALGO_POPC && C * kk > kTcMaxK) return BT_ERR_UNSUPPORTED;
    // the plan bt_tune_conv2d kept for this geometry, unless one is forced already
    ConvChoice kept{};
    const bool use_kept = conv_forced() == nullptr && conv_lookup(g, w_code, out_dtype, kept);
    if (use_kept) conv_force(&kept);
    struct Unforce {
        bool on;
        ~Unforce() {
            if (on) conv_force(nullptr);
        }
    } unforce{use_kept};

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t need = bt_binary_conv2d_workspace(B, C, H, W, kernel_size, stride, padding, dilation, x_dtype,
                                                   w_code);
    const bool implicit = run != BT_ALGO_POPC && x_dtype != BT_PACKED_IM2COL && conv_implicit_applies(g, w_code);
    // one kernel from x where the contraction can pack its own input
    const bool fused = implicit && float_in(x_dtype) && conv_fused_applies(g, w_code, x_dtype) &&
                       (bias_len == 0 || aligned(bias_a, 4));
    const bool needs_ws = (float_in(x_dtype) && !fused) || (x_dtype == BT_PACKED && run != BT_ALGO_POPC && !implicit);
    if (needs_ws && need == 0) return BT_ERR_UNSUPPORTED;      // beyond the sizes the query serves
    if (needs_ws && (workspace == nullptr || workspace_bytes < need)) return BT_ERR_WORKSPACE;
    if (needs_ws && !aligned(workspace, 256)) return BT_ERR_ALIGNMENT;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const int64_t rbc = row_bytes(C, w_code);
    const float alpha = alpha_of(scale_a, scale_w);
    unsigned int *err = device_error_word();
    if (err == nullptr) return BT_ERR_CUDA;
    if (x_dtype == BT_PACKED_IM2COL)
        return from_cuda(launch_tc_conv(static_cast<const uint8_t *>(x), static_cast<const uint8_t *>(weight), w_code,
                                        g, alpha, out, out_dtype, err, s, scales));
    if (fused) {
        const cudaError_t e = launch_tc_conv_fused(x, x_dtype, bias_len > 0 ? bias_a : nullptr, bias_len,
                                                   static_cast<const uint8_t *>(weight), w_code, g, alpha, out,
                                                   out_dtype, err, s, scales);
        if (e == cudaErrorNotSupported) return BT_ERR_UNSUPPORTED;
        return from_cuda(e);
    }
    if (implicit) {
        // pack to channel-packed NHWC pixels (unless given), then the
        // implicit-im2col contraction reads them in place
        const void *xp = x;
        if (x_dtype != BT_PACKED) {
            if (launch_pack_nhwc(x, x_dtype, B, C, H * W, bias_a, bias_len, w_code, ws, s) != cudaSuccess)
                return BT_ERR_CUDA;
            xp = ws;
        }
        const cudaError_t e = launch_tc_conv_implicit(static_cast<const uint8_t *>(xp),
                                                      static_cast<const uint8_t *>(weight), w_code, g, alpha, out,
                                                      out_dtype, err, s, scales, x_dtype != BT_PACKED);
        if (e == cudaErrorNotSupported) return BT_ERR_UNSUPPORTED;
        return from_cuda(e);
    }
    uint8_t *rows = ws + (x_dtype == BT_PACKED ? 0 : round_up(static_cast<size_t>(B * H * W * rbc), 256));
    if (run != BT_ALGO_POPC && x_dtype != BT_PACKED) {
        // one pass from x to the im2col rows, where the staged unfold applies
        const cudaError_t e = launch_pack_im2col(x, x_dtype, g, bias_a, bias_len, w_code, rows, false, s);
        if (e == cudaSuccess)
            return from_cuda(launch_tc_conv(rows, static_cast<const uint8_t *>(weight), w_code, g, alpha, out,
                                            out_dtype, err, s, scales));
        if (e != cudaErrorNotSupported) return BT_ERR_CUDA;
    }
    const void *xp = x;
    if (x_dtype != BT_PACKED) {
        cudaError_t e = launch_pack_nhwc(x, x_dtype, B, C, H * W, bias_a, bias_len, w_code, ws, s);
        if (e != cudaSuccess) return BT_ERR_CUDA;
        xp = ws;
    }
    if (run == BT_ALGO_POPC)
        return from_cuda(launch_popc_conv(static_cast<const uint32_t *>(xp), static_cast<const uint32_t *>(weight),
                                          g, alpha, out, out_dtype, s, scales));
    cudaError_t e = launch_im2col_rows(static_cast<const uint8_t *>(xp), g, rbc, rows, s);
    if (e != cudaSuccess) return BT_ERR_CUDA;
    return from_cuda(launch_tc_conv(rows, static_cast<const uint8_t *>(weight), w_code, g, alpha, out, out_dtype, err,
                                    s, scales));
}
}  // namespace

bt_status bt_binary_conv2d(const void *x, bt_dtype x_dtype, const void *weight, bt_code w_code,
                           int64_t B, int64_t C, int64_t H, int64_t W, int64_t O, int kernel_size,
                           int stride, int padding, int dilation, float scale_a, float scale_w,
                           const float *bias_a, int64_t bias_len, void *out, bt_dtype out_dtype,
                           bt_algo algo, void *workspace, size_t workspace_bytes, bt_stream stream) {
    if (algo == BT_ALGO_TUNE) {
        algo = BT_ALGO_AUTO;
        // a geometry with implicit plans to choose from and none kept yet: tune it
        // (the last timed call leaves this call's result in out)
        if ((w_code == BT_CODE_E4M3 || w_code == BT_CODE_E2M1) && x_dtype != BT_PACKED_IM2COL && valid_out(out_dtype) &&
            B >= 1 && C >= 1 && H >= 1 && W >= 1 && O >= 1 && kernel_size >= 1 && kernel_size <= 64 &&
            stride >= 1 && padding >= 0 && dilation >= 1 && H <= (1 << 20) && W <= (1 << 20) && C <= kTcMaxK &&
            C * kernel_size * kernel_size <= kTcMaxK) {
            ConvGeom g{B, C, H, W, O, 0, 0, kernel_size, stride, padding, dilation};
            g.Ho = conv_out(H, kernel_size, stride, padding, dilation);
            g.Wo = conv_out(W, kernel_size, stride, padding, dilation);
            ConvChoice kept{};
            if (g.Ho >= 1 && g.Wo >= 1 && conv_implicit_applies(g, w_code) &&
                !conv_lookup(g, w_code, out_dtype, kept) && !stream_capturing(reinterpret_cast<cudaStream_t>(stream))) {
                bt_tune_conv_result r;
                return bt_tune_conv2d(x, x_dtype, weight, w_code, B, C, H, W, O, kernel_size, stride, padding,
                                      dilation, scale_a, scale_w, bias_a, bias_len, out, out_dtype, workspace,
                                      workspace_bytes, kAutoTuneReps, stream, &r);
            }
        }
    }
    return conv_impl(x, x_dtype, weight, w_code, B, C, H, W, O, kernel_size, stride, padding, dilation, scale_a,
                     scale_w, nullptr, bias_a, bias_len, out, out_dtype, algo, workspace, workspace_bytes, stream);
}

bt_status bt_binary_conv2d_dscale(const void *x, bt_dtype x_dtype, const void *weight, bt_code w_code, int64_t B,
                                  int64_t C, int64_t H, int64_t W, int64_t O, int kernel_size, int stride,
                                  int padding, int dilation, const float *scales, const float *bias_a,
                                  int64_t bias_len, void *out, bt_dtype out_dtype, bt_algo algo, void *workspace,
                                  size_t workspace_bytes, bt_stream stream) {
    if (scales == nullptr) return BT_ERR_INVALID_ARG;
    return conv_impl(x, x_dtype, weight, w_code, B, C, H, W, O, kernel_size, stride, padding, dilation, 1.0f, 1.0f,
                     scales, bias_a, bias_len, out, out_dtype, algo, workspace, workspace_bytes, stream);
}

bt_status bt_binary_conv2d_dscale_init(const void *x, bt_dtype x_dtype, const void *weight, bt_code w_code,
                                       int64_t B, int64_t C, int64_t H, int64_t W, int64_t O, int kernel_size,
                                       int stride, int padding, int dilation, float *scales, float factor,
                                       bt_dtype scale_dtype, const float *bias_a, int64_t bias_len, void *out,
                                       bt_dtype out_dtype, bt_algo algo, void *workspace, size_t workspace_bytes,
                                       bt_stream stream) {
    if (scales == nullptr || !float_in(x_dtype) || !float_in(scale_dtype)) return BT_ERR_INVALID_ARG;
    if (!(std::isfinite(factor) && factor > 0.0f)) return BT_ERR_INVALID_ARG;
    if (!valid_code(w_code) || !valid_out(out_dtype)) return BT_ERR_INVALID_ARG;
    if (B < 0 || C < 1 || H < 1 || W < 1 || O < 0) return BT_ERR_INVALID_ARG;
    if (kernel_size < 1 || stride < 1 || padding < 0 || dilation < 1) return BT_ERR_INVALID_ARG;
    if (!(bias_len == 0 || bias_len == 1 || bias_len == C) || (bias_len > 0 && bias_a == nullptr))
        return BT_ERR_INVALID_ARG;
    if (conv_out(H, kernel_size, stride, padding, dilation) < 1 || conv_out(W, kernel_size, stride, padding, dilation) < 1)
        return BT_ERR_INVALID_ARG;
    if (B == 0 || O == 0) return BT_OK;
    if (x == nullptr || weight == nullptr || out == nullptr) return BT_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(weight, 16) || !aligned(out, 16) || !aligned(scales, 8)) return BT_ERR_ALIGNMENT;
    if (B > (int64_t(1) << 30) || C > kMaxK || H > (1 << 20) || W > (1 << 20)) return BT_ERR_UNSUPPORTED;
    // workspace: the packed NHWC pixels, then what the contraction of packed
    // pixels needs (the im2col rows of the explicit unfold, or nothing)
    const size_t need = bt_binary_conv2d_workspace(B, C, H, W, kernel_size, stride, padding, dilation, x_dtype,
                                                   w_code);
    if (need == 0) return BT_ERR_UNSUPPORTED;
    if (workspace == nullptr || workspace_bytes < need) return BT_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return BT_ERR_ALIGNMENT;
    const size_t pix = round_up(static_cast<size_t>(B * H * W * row_bytes(C, w_code)), 256);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err = cudaSuccess;
    double *acc = fused_abs_sum_accumulator(&err);
    if (acc == nullptr || cudaMemsetAsync(acc, 0, sizeof(double), s) != cudaSuccess) return BT_ERR_CUDA;
    cudaError_t e = launch_pack_nhwc_sum(x, x_dtype, B, C, H * W, bias_a, bias_len, w_code, workspace, acc, s);
    if (e == cudaErrorNotSupported) {
        e = launch_pack_nhwc(x, x_dtype, B, C, H * W, bias_a, bias_len, w_code, workspace, s);
        if (e == cudaSuccess) e = launch_abs_sum(x, x_dtype, B * C * H * W, acc, s);
    }
    if (e != cudaSuccess) return BT_ERR_CUDA;
    if (launch_scale_finish(acc, B * C * H * W, factor, x_dtype, scale_dtype, scales, s) != cudaSuccess)
        return BT_ERR_CUDA;
    uint8_t *rest = static_cast<uint8_t *>(workspace) + pix;
    return conv_impl(workspace, BT_PACKED, weight, w_code, B, C, H, W, O, kernel_size, stride, padding, dilation, 1.0f,
                     1.0f, scales, nullptr, 0, out, out_dtype, algo, need > pix ? rest : nullptr,
                     need > pix ? workspace_bytes - pix : 0, stream);
}

int bt_conv2d_single_pass(int64_t B, int64_t C, int64_t H, int64_t W, int kernel_size, int stride, int padding,
                          int dilation, bt_dtype x_dtype, bt_code code) {
    if (!float_in(x_dtype) || (code != BT_CODE_E4M3 && code != BT_CODE_E2M1)) return 0;
    if (B < 1 || C < 1 || H < 1 || W < 1 || kernel_size < 1 || stride < 1 || padding < 0 || dilation < 1) return 0;
    if (H > (1 << 20) || W > (1 << 20) || kernel_size > 64 || padding > (1 << 20) || stride > (1 << 20) ||
        dilation > (1 << 10) || C > kTcMaxK || C * kernel_size * kernel_size > kTcMaxK)
        return 0;
    ConvGeom g{B, C, H, W, 0, 0, 0, kernel_size, stride, padding, dilation};
    g.Ho = conv_out(H, kernel_size, stride, padding, dilation);
    g.Wo = conv_out(W, kernel_size, stride, padding, dilation);
    if (g.Ho < 1 || g.Wo < 1) return 0;
    bool kept_fused = false;
    if (conv_forced() == nullptr && conv_kept_fused(g, code, kept_fused)) {
        // the route bt_tune_conv2d kept for this geometry
        const ConvChoice f{-1, 0, 0, kept_fused ? 1 : 0, 0};
        conv_force(&f);
        const bool fused = conv_fused_applies(g, code, x_dtype);
        conv_force(nullptr);
        if (fused) return 2;
    } else if (conv_fused_applies(g, code, x_dtype)) {
        return 2;                                          // one kernel from x
    }
    if (conv_implicit_applies(g, code)) return 0;      // packed pixels, contracted in place
    return unfold_single_pass(g, x_dtype, code) ? 1 : 0;
}

bt_status bt_pack_im2col(const void *x, bt_dtype x_dtype, int64_t B, int64_t C, int64_t H, int64_t W,
                         int kernel_size, int stride, int padding, int dilation, const float *bias,
                         int64_t bias_len, bt_code code, void *out, bt_stream stream) {
    if (!float_in(x_dtype) || (code != BT_CODE_E4M3 && code != BT_CODE_E2M1)) return BT_ERR_INVALID_ARG;
    if (B < 0 || C < 1 || H < 1 || W < 1) return BT_ERR_INVALID_ARG;
    if (kernel_size < 1 || stride < 1 || padding < 0 || dilation < 1) return BT_ERR_INVALID_ARG;
    if (!(bias_len == 0 || bias_len == 1 || bias_len == C)) return BT_ERR_INVALID_ARG;
    if (bias_len > 0 && bias == nullptr) return BT_ERR_INVALID_ARG;
    ConvGeom g{B, C, H, W, 0, 0, 0, kernel_size, stride, padding, dilation};
    g.Ho = conv_out(H, kernel_size, stride, padding, dilation);
    g.Wo = conv_out(W, kernel_size, stride, padding, dilation);
    if (g.Ho < 1 || g.Wo < 1) return BT_ERR_INVALID_ARG;
    const int64_t kk = static_cast<int64_t>(kernel_size) * kernel_size;
    if (C > kTcMaxK || kernel_size > 64 || C * kk > kTcMaxK || H > (1 << 20) || W > (1 << 20) || padding > (1 << 20) ||
        stride > (1 << 20) || dilation > (1 << 10))
        return BT_ERR_UNSUPPORTED;
    if (B == 0) return BT_OK;
    if (B > int64_t(65535) * 128 || g.Ho * g.Wo > int64_t(65535) * 128 || B * g.Ho * g.Wo > int64_t(65535) * 128)
        return BT_ERR_UNSUPPORTED;
    if (x == nullptr || out == nullptr) return BT_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(out, 16) || (bias && !aligned(bias, 4))) return BT_ERR_ALIGNMENT;
    return from_cuda(launch_pack_im2col(x, x_dtype, g, bias, bias_len, code, static_cast<uint8_t *>(out), true,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
// The call times bt_tune_linear / bt_tune_conv2d measured per device, layer
// kind and problem size (M, N, K), one per code (the last timing of each, over
// whatever output dtype it was run with); bt_plan takes the shortest.
struct CodeKey {
    int dev, op;
    int64_t M, N, K;
    bool operator<(const CodeKey &o) const {
        if (dev != o.dev) return dev < o.dev;
        if (op != o.op) return op < o.op;
        if (M != o.M) return M < o.M;
        if (N != o.N) return N < o.N;
        return K < o.K;
    }
};
struct CodeTime {
    float us[3];        // per code, < 0 when not measured
};
std::mutex g_code_mu;
std::map<CodeKey, CodeTime> g_code_times;

CodeKey code_key(bt_op op, int64_t M, int64_t N, int64_t K) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
    return CodeKey{dev, static_cast<int>(op), M, N, K};
}

void record_code_time(bt_op op, int64_t M, int64_t N, int64_t K, bt_code code, float us) {
    std::lock_guard<std::mutex> lock(g_code_mu);
    auto ins = g_code_times.insert({code_key(op, M, N, K), CodeTime{{-1.0f, -1.0f, -1.0f}}});
    ins.first->second.us[static_cast<int>(code)] = us;
}

bool measured_code(bt_op op, int64_t M, int64_t N, int64_t K, bt_code &code) {
    std::lock_guard<std::mutex> lock(g_code_mu);
    if (g_code_times.empty()) return false;
    auto it = g_code_times.find(code_key(op, M, N, K));
    if (it == g_code_times.end()) return false;
    int best = -1;
    for (int c = 0; c < 3; ++c)
        if (it->second.us[c] >= 0.0f && (best < 0 || it->second.us[c] < it->second.us[best])) best = c;
    if (best < 0) return false;
    code = static_cast<bt_code>(best);
    return true;
}

// Mean time of `reps` calls of `run` on stream s (after one untimed call),
// in microseconds; negative when a call fails.
float time_calls(const std::function<bt_status()> &run, int reps, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1, bt_status &st) {
    st = run();
    if (st != BT_OK) return -1.0f;
    if (cudaEventRecord(e0, s) != cudaSuccess) return st = BT_ERR_CUDA, -1.0f;
    for (int i = 0; i < reps; ++i)
        if ((st = run()) != BT_OK) return -1.0f;
    if (cudaEventRecord(e1, s) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess) return st = BT_ERR_CUDA, -1.0f;
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess) return st = BT_ERR_CUDA, -1.0f;
    return 1000.0f * ms / static_cast<float>(reps);
}
}  // namespace

bt_status bt_tune_linear(const void *x, bt_dtype x_dtype, const void *weight, bt_code w_code, int64_t M, int64_t N,
                         int64_t K, float scale_a, float scale_w, const float *bias_a, int64_t bias_len, void *out,
                         bt_dtype out_dtype, void *workspace, size_t workspace_bytes, int reps, bt_stream stream,
                         bt_tune_result *result) {
    if (result == nullptr || reps < 1 || reps > 10000) return BT_ERR_INVALID_ARG;
    *result = bt_tune_result{};
    result->code = w_code;
    if (M < 1 || N < 1) {
        // nothing to time: a zero-size call is a no-op (or its argument error)
        return linear_impl(x, x_dtype, weight, w_code, M, N, K, scale_a, scale_w, nullptr, bias_a, bias_len, out,
                           out_dtype, BT_ALGO_AUTO, workspace, workspace_bytes, stream);
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return BT_ERR_CUDA;
    if (cap != cudaStreamCaptureStatusNone) return BT_ERR_UNSUPPORTED;       // timing needs real launches
    auto run = [&] {
        return linear_impl(x, x_dtype, weight, w_code, M, N, K, scale_a, scale_w, nullptr, bias_a, bias_len, out,
                           out_dtype, BT_ALGO_AUTO, workspace, workspace_bytes, stream);
    };
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess) return BT_ERR_CUDA;
    if (cudaEventCreate(&e1) != cudaSuccess) {
        cudaEventDestroy(e0);
        return BT_ERR_CUDA;
    }
    bt_status st = BT_OK;
    float best = -1.0f;
    if (w_code == BT_CODE_BITS) {
        // one kernel for this code: time it
        best = time_calls(run, reps, s, e0, e1, st);
        result->candidates = 1;
        result->us_model = best;
    } else {
        TcTileChoice cand[24];
        const int n = tc_linear_candidates(M, N, K, w_code, out_dtype, cand, 24);
        TcTileChoice win{};
        for (int i = 0; i < n; ++i) {
            tc_linear_force(&cand[i]);
            const float us = time_calls(run, reps, s, e0, e1, st);
            tc_linear_force(nullptr);
            if (us < 0.0f) break;
            ++result->candidates;
            if (i == 0) result->us_model = us;
            // another shape replaces the one kept so far (the model's own
            // first) only when it measures more than 1 % faster: timing noise
            // does not move the choice
            if (best < 0.0f || us < 0.99f * best) {
                best = us;
                win = cand[i];
            }
        }
        if (st == BT_OK && n == 0) st = run();          // argument errors of a call with no candidate
        if (st == BT_OK && best >= 0.0f) {
            tc_linear_remember(M, N, K, w_code, out_dtype, win);
            result->pair = win.pair;
            result->bn = win.bn;
            result->slices_per_stage = win.d;
            result->epilogue_warps = win.epi;
        }
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (st != BT_OK) return st;
    result->us = best;
    if (best >= 0.0f) record_code_time(BT_OP_LINEAR, M, N, K, w_code, best);
    return BT_OK;
}

bt_status bt_tune_conv2d(const void *x, bt_dtype x_dtype, const void *weight, bt_code w_code, int64_t B, int64_t C,
                         int64_t H, int64_t W, int64_t O, int kernel_size, int stride, int padding, int dilation,
                         float scale_a, float scale_w, const float *bias_a, int64_t bias_len, void *out,
                         bt_dtype out_dtype, void *workspace, size_t workspace_bytes, int reps, bt_stream stream,
                         bt_tune_conv_result *result) {
    if (result == nullptr || reps < 1 || reps > 10000) return BT_ERR_INVALID_ARG;
    *result = bt_tune_conv_result{};
    result->code = w_code;
    auto run = [&] {
        return conv_impl(x, x_dtype, weight, w_code, B, C, H, W, O, kernel_size, stride, padding, dilation, scale_a,
                         scale_w, nullptr, bias_a, bias_len, out, out_dtype, BT_ALGO_AUTO, workspace,
                         workspace_bytes, stream);
    };
    // argument errors and empty problems: what the call itself answers
    const int64_t Ho = conv_out(H, kernel_size, stride, padding, dilation);
    const int64_t Wo = conv_out(W, kernel_size, stride, padding, dilation);
    if (!valid_code(w_code) || B < 1 || O < 1 || C < 1 || H < 1 || W < 1 || kernel_size < 1 || stride < 1 ||
        padding < 0 || dilation < 1 || Ho < 1 || Wo < 1)
        return run();
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return BT_ERR_CUDA;
    if (cap != cudaStreamCaptureStatusNone) return BT_ERR_UNSUPPORTED;       // timing needs real launches
    ConvGeom g{B, C, H, W, O, Ho, Wo, kernel_size, stride, padding, dilation};
    ConvChoice cand[64];
    const int n = (x_dtype == BT_PACKED_IM2COL || w_code == BT_CODE_BITS)
                      ? 0 : conv_candidates(g, w_code, x_dtype, out_dtype, cand, 64);
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess) return BT_ERR_CUDA;
    if (cudaEventCreate(&e1) != cudaSuccess) {
        cudaEventDestroy(e0);
        return BT_ERR_CUDA;
    }
    bt_status st = BT_OK;
    float best = -1.0f;
    if (n == 0) {
        // one route for this code and geometry: time it
        best = time_calls(run, reps, s, e0, e1, st);
        result->candidates = st == BT_OK ? 1 : 0;
        result->us_model = best;
    } else {
        ConvChoice win{};
        for (int i = 0; i < n; ++i) {
            conv_force(&cand[i]);
            const float us = time_calls(run, reps, s, e0, e1, st);
            conv_force(nullptr);
            if (us < 0.0f) break;
            ++result->candidates;
            if (i == 0) result->us_model = us;
            // as for the linear layer: a plan replaces the planner's only when > 1 % faster
            if (best < 0.0f || us < 0.99f * best) {
                best = us;
                win = cand[i];
            }
        }
        if (st == BT_OK && best >= 0.0f) {
            conv_remember(g, w_code, out_dtype, win);
            result->pair = win.pair;
            result->weights_resident = win.plan == 'R' ? 1 : 0;
            result->pixel_stages = win.bst;
            result->fused = win.fused;
            result->band_split = win.split > 1 ? win.split : 1;
        }
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (st != BT_OK) return st;
    result->us = best;
    if (best >= 0.0f) record_code_time(BT_OP_CONV2D, B * Ho * Wo, O, C * kernel_size * kernel_size, w_code, best);
    return BT_OK;
}

bt_status bt_conv2d_plan_info(int64_t B, int64_t C, int64_t H, int64_t W, int64_t O, int kernel_size, int stride,
                              int padding, int dilation, bt_code code, bt_dtype out_dtype, int sms, int pair, int split,
                              bt_conv_plan_info *info) {
    if (info == nullptr) return BT_ERR_INVALID_ARG;
    *info = bt_conv_plan_info{};
    if ((code != BT_CODE_E4M3 && code != BT_CODE_E2M1) || !valid_out(out_dtype)) return BT_ERR_INVALID_ARG;
    if (B < 1 || C < 1 || H < 1 || W < 1 || O < 1 || kernel_size < 1 || stride < 1 || padding < 0 || dilation < 1)
        return BT_ERR_INVALID_ARG;
    if (sms < 1 || pair < -1 || pair > 1 || split < 1) return BT_ERR_INVALID_ARG;
    if (B > (int64_t(1) << 30) || C > kMaxK || H > (1 << 20) || W > (1 << 20) || kernel_size > 64 ||
        padding > (1 << 20) || stride > (1 << 20) || dilation > (1 << 10))
        return BT_ERR_INVALID_ARG;
    ConvGeom g{B, C, H, W, O, 0, 0, kernel_size, stride, padding, dilation};
    g.Ho = conv_out(H, kernel_size, stride, padding, dilation);
    g.Wo = conv_out(W, kernel_size, stride, padding, dilation);
    if (g.Ho < 1 || g.Wo < 1) return BT_ERR_INVALID_ARG;
    conv_plan_query(g, code, out_dtype == BT_BF16 || out_dtype == BT_F16 ? 2 : 4, sms, pair, split, *info);
    return BT_OK;
}

void bt_tune_reset(void) {
    tc_linear_forget();
    conv_forget();
    std::lock_guard<std::mutex> lock(g_code_mu);
    g_code_times.clear();
}

bt_status bt_plan(bt_op op, int64_t M, int64_t N, int64_t K, bt_code *code, bt_algo *algo) {
    if (code == nullptr || algo == nullptr || M < 1 || N < 1 || K < 1) return BT_ERR_INVALID_ARG;
    if (op != BT_OP_LINEAR && op != BT_OP_CONV2D) return BT_ERR_INVALID_ARG;
    bt_code c = BT_CODE_BITS;
    const char *force = std::getenv("BT_FORCE_ALGO");
    if (force != nullptr && std::strcmp(force, "popc") == 0) c = BT_CODE_BITS;
    else if (force != nullptr && std::strcmp(force, "e4m3") == 0) c = BT_CODE_E4M3;
    else if (force != nullptr && std::strcmp(force, "e2m1") == 0) c = BT_CODE_E2M1;
    else if (measured_code(op, M, N, K, c)) {
        // the fastest code bt_tune_linear / bt_tune_conv2d measured for this size
    } else c = (K <= kTcMaxK && tc_available()) ? BT_CODE_E2M1 : BT_CODE_BITS;
    *code = c;
    *algo = algo_for_code(c);
    return BT_OK;
}

bt_status bt_set_wait_timeout(uint64_t ns) {
    if (ns > 60ull * 1000000000ull) return BT_ERR_INVALID_ARG;
    g_wait_limit_ns.store(ns == 0 ? kWaitNs : ns, std::memory_order_relaxed);
    return BT_OK;
}

bt_status bt_device_status(bt_stream stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return BT_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word)) != cudaSuccess) return BT_ERR_CUDA;
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) return BT_ERR_CUDA;
        return BT_ERR_TIMEOUT;
    }
    return BT_OK;
}

}  // extern "C"
