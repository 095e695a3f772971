/*
 * bt.h -- C ABI of libbt: the binarized linear and conv2d forward on one
 * NVIDIA GB300 (sm_103a).
 *
 * The method (bitorch-engine: BinaryConv2dCutlass / BinaryConv2dForward,
 * BinaryLinearCuda / BinaryLinearForward):
 *   1. shift      a = x + bias_a            (set_activation, "learnable shift input")
 *   2. binarize   sa = +1 if a >= 0 else -1, sw = +1 if W >= 0 else -1
 *   3. contract   dot = sum_k sa*sw = K - 2*popcount(bits(sa) XOR bits(sw))
 *                 (a convolution through an implicit im2col)
 *   4. scale      y = fp32(dot * alpha), alpha = fp32(scale_a * scale_w)
 *                 (the native forward receives scale_a.item()*scale_w.item())
 *   5. cast       out = y.to(x.dtype)        (BinaryConv2dForward.forward)
 *
 * Conventions for every call:
 *   - Pointers named "device" are CUDA device (or managed) memory; all work is
 *     enqueued asynchronously on `stream` (NULL = the legacy default stream).
 *     The caller owns every buffer; the library allocates nothing and keeps no
 *     pointer after a call returns.
 *   - Tensors are dense and contiguous (row-major / NCHW as stated). Device
 *     pointers must be 16-byte aligned; the workspace 256-byte aligned.
 *   - Arguments are validated on the host before anything is launched; a
 *     failed check returns an error status and launches nothing.
 *   - A launch failure returns BT_ERR_CUDA. Kernels never trap: a bounded
 *     wait that runs out records BT_ERR_TIMEOUT in a device error word and the
 *     kernel returns; bt_device_status() reports it.
 *   - No call aborts the process.
 *
 * Binarization rule: +1 where x + bias >= 0 (the sum in IEEE fp32 without
 * flushing subnormals, whose sign is the sign of the exact sum), else -1;
 * -0.0 gives +1 and NaN gives -1. Weights use the same rule without a shift.
 * The shift is added, as BinaryConv2dCutlass.set_activation does
 * (x + bias_a.view(1,-1,1,1)); for a subtracted shift (x - b), pass -b.
 */
#ifndef BT_H
#define BT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st *bt_stream;

typedef enum {
    BT_OK = 0,
    BT_ERR_INVALID_ARG = -1,   /* null pointer, bad size, bad scale, bad enum value */
    BT_ERR_UNSUPPORTED = -2,   /* valid request this build cannot serve (e.g. algo vs code) */
    BT_ERR_ALIGNMENT = -3,     /* a pointer misses its required alignment */
    BT_ERR_WORKSPACE = -4,     /* workspace missing or smaller than the query says */
    BT_ERR_CUDA = -5,          /* a CUDA runtime call or launch failed */
    BT_ERR_TIMEOUT = -6        /* a kernel's bounded wait ran out (device error word) */
} bt_status;

/* Element types. BT_PACKED is an input already packed in the weight's code;
 * BT_PACKED_IM2COL a convolution input already unfolded by bt_pack_im2col. */
typedef enum {
    BT_F32 = 0,
    BT_BF16 = 1,
    BT_F16 = 2,
    BT_I32 = 3,            /* output only: the raw integer dot products */
    BT_PACKED = 4,         /* input only */
    BT_PACKED_IM2COL = 5   /* input only (bt_binary_conv2d, codes E4M3 / E2M1) */
} bt_dtype;

/*
 * Packed operand encodings ("bit-packing" of bitorch-engine's w_pack /
 * generate_quantized_weight, there with 8-bit words). A packed row of k
 * elements occupies bt_packed_row_bytes(k, code) bytes (BITS: rounded up to
 * 16 bytes; E4M3 / E2M1: rounded up to 64 bytes); every position after the
 * last element is 0.
 *
 *   BT_CODE_BITS  1 bit per element in little-endian uint32 words: bit j of
 *                 word w holds element 32*w + j; 1 means +1, 0 means -1.
 *                 Contracted by XOR + popcount: dot = k - 2*popc(a ^ w).
 *   BT_CODE_E4M3  1 byte per element, the FP8 E4M3 value +1.0 (0x38) or
 *                 -1.0 (0xB8); padding is 0x00 (0.0).
 *   BT_CODE_E2M1  4 bits per element, the FP4 E2M1 value +1.0 (0x2) or -1.0
 *                 (0xA), element 2i in the low nibble of byte i; padding 0.
 *
 * The E4M3 / E2M1 encodings feed the tcgen05 tensor cores; products of +1/-1
 * codes are +1/-1 and the sums are integers, so dot is the same integer as
 * with BITS. A padded or zero-filled position contributes 0.
 */
typedef enum {
    BT_CODE_BITS = 0,
    BT_CODE_E4M3 = 1,
    BT_CODE_E2M1 = 2
} bt_code;

typedef enum {
    BT_LAYOUT_ROWS = 0,          /* [R, K] row-major -> [R, row_bytes(K)] */
    BT_LAYOUT_NCHW_TO_NHWC = 1   /* [B, C, H, W] -> [B, H, W, row_bytes(C)] (channel-packed) */
} bt_layout;

/*
 * Contraction kernels (the BMM type of BinaryLinearCuda, whose default
 * BMM.ADAPTIVE picks one; here BT_ALGO_AUTO does, and BT_ALGO_TUNE does by
 * measurement).
 */
typedef enum {
    BT_ALGO_AUTO = 0,        /* the kernel for the weight's code chosen by bt_plan() */
    BT_ALGO_POPC = 1,        /* CUDA cores: XOR + popcount, code BITS */
    BT_ALGO_TC_E4M3 = 2,     /* tcgen05 kind::f8f6f4 on +1/-1 E4M3, code E4M3 */
    BT_ALGO_TC_E2M1 = 3,     /* tcgen05 kind::mxf4 on +1/-1 E2M1 (unit block scales), code E2M1 */
    BT_ALGO_TUNE = 4         /* AUTO, measured: bt_binary_linear / bt_binary_conv2d only. The first
                                call of a size (on this device, with this code and output dtype)
                                that has launch shapes or plans to choose from runs bt_tune_linear /
                                bt_tune_conv2d (3 timed calls per candidate; it blocks the calling
                                thread) and returns with that call's result in out; later calls take
                                the kept shape or plan. Inside a stream capture, for BT_CODE_BITS and
                                where the convolution has one route, it runs as AUTO. */
} bt_algo;

typedef enum { BT_OP_LINEAR = 0, BT_OP_CONV2D = 1 } bt_op;

/* Library version as 10000*major + 100*minor + patch. */
int bt_version(void);

/* Static text for a status code; never NULL. */
const char *bt_status_string(bt_status status);

/* Bytes of one packed row of k elements in `code` (BITS: a multiple of 16;
 * E4M3 / E2M1: a multiple of 64); -1 for k < 0 or an unknown code. */
int64_t bt_packed_row_bytes(int64_t k, bt_code code);

/*
 * bt_pack_sign -- fused shift + sign + pack (BinaryConv2dCutlass.set_activation
 * followed by the native binarization; w_pack for weights).
 *
 *   x        device, x_dtype in {BT_F32, BT_BF16, BT_F16}, dense:
 *              ROWS:          [d0=R, d1=K]            (d2, d3 ignored)
 *              NCHW_TO_NHWC:  [d0=B, d1=C, d2=H, d3=W] (OIHW weights: B=O, H=W=k)
 *   bias     device fp32 or NULL; bias_len 0 (none), 1 (one scalar) or d1
 *            (one per column of ROWS / per channel of NCHW).
 *   out      device, ROWS: [R, bt_packed_row_bytes(K, code)] bytes;
 *            NCHW_TO_NHWC: [B, H, W, bt_packed_row_bytes(C, code)] bytes.
 * Errors: BT_ERR_INVALID_ARG for null x/out, d0..d3 < 1 (d0 = 0 rows is
 * allowed and does nothing), a bad bias_len or enum; BT_ERR_ALIGNMENT when x or
 * out is not 16-byte aligned.
 */
bt_status bt_pack_sign(const void *x, bt_dtype x_dtype, bt_layout layout,
                       int64_t d0, int64_t d1, int64_t d2, int64_t d3,
                       const float *bias, int64_t bias_len,
                       bt_code code, void *out, bt_stream stream);

/*
 * bt_pack_im2col -- fused shift + sign + pack + unfold of a convolution's
 * input (BinaryConv2dCutlass.set_activation and binarization, then the unfold
 * of banghao.live/blog/9 section 2, MyConv2d.forward, on packed codes): the
 * matrix a tensor-core bt_binary_conv2d contracts with the weights.
 *
 *   x        device NCHW [B, C, H, W] in x_dtype (BT_F32 / BF16 / F16).
 *   bias     device fp32 or NULL; bias_len 0, 1 or C (per input channel).
 *   code     BT_CODE_E4M3 or BT_CODE_E2M1.
 *   out      device [B*Ho*Wo, k*k*bt_packed_row_bytes(C, code)] bytes, 16-byte
 *            aligned; Ho, Wo as in bt_binary_conv2d. Row (b, ho, wo) holds, for
 *            each tap (kh, kw) in turn, the packed input pixel
 *            (ho*s - p + kh*d, wo*s - p + kw*d) of image b, all zero codes
 *            where that pixel is in the padding.
 * Errors: BT_ERR_INVALID_ARG for null pointers, bad sizes, a bad bias_len or
 * code; BT_ERR_ALIGNMENT when x or out is not 16-byte aligned; BT_ERR_UNSUPPORTED
 * beyond the sizes bt_binary_conv2d serves. B = 0 does nothing.
 */
bt_status bt_pack_im2col(const void *x, bt_dtype x_dtype, int64_t B, int64_t C, int64_t H, int64_t W,
                         int kernel_size, int stride, int padding, int dilation,
                         const float *bias, int64_t bias_len, bt_code code, void *out, bt_stream stream);

/*
 * bt_conv2d_single_pass -- how bt_binary_conv2d, given a 16-byte aligned float
 * x of this geometry and a tensor-core code, splits its own work:
 *   2  one kernel from x: the tensor-core convolution packs x itself (shift,
 *      sign, channel packing into its shared-memory pixel stages) and needs
 *      no workspace -- where the implicit-im2col plan applies, every channel
 *      plane (H * W values of x_dtype) is a multiple of 16 bytes and the
 *      environment sets BT_CONV_FUSED=1, or bt_tune_conv2d kept that route
 *      for the geometry (slower than route 0 on the ResNet layers measured,
 *      so not the default);
 *   1  the im2col rows built in one pass from x (the staged form of
 *      bt_pack_im2col), then the contraction of those rows;
 *   0  the pixels packed to NHWC (bt_pack_sign NCHW_TO_NHWC), then the
 *      contraction of the packed pixels (in place, or after an unfold); also
 *      for BITS and for invalid arguments.
 * The result is the same on every route; this tells a caller which public
 * calls reproduce the library's own launches (the one call on float x; or
 * bt_pack_im2col + BT_PACKED_IM2COL; or bt_pack_sign + BT_PACKED).
 * (BinaryConv2dForward.forward of bitorch-engine's layer module is one native
 * call from x to the scaled output.)
 */
int bt_conv2d_single_pass(int64_t B, int64_t C, int64_t H, int64_t W, int kernel_size, int stride,
                          int padding, int dilation, bt_dtype x_dtype, bt_code code);

/* Workspace bytes bt_binary_linear needs (0 when x is BT_PACKED). */
size_t bt_binary_linear_workspace(int64_t M, int64_t K, bt_dtype x_dtype, bt_code code);

/*
 * bt_binary_linear -- out = cast(fp32(dot * fp32(scale_a*scale_w))),
 * dot[m,n] = sum_k sign(x[m,k] + bias) * sign(W[n,k])
 * (BinaryLinearForward.forward(input, weight, bmm_type, scale_a, scale_w)).
 *
 *   x          device [M, K] in x_dtype (BT_F32/BF16/F16), or BT_PACKED:
 *              [M, bt_packed_row_bytes(K, w_code)] already in w_code.
 *   weight     device [N, bt_packed_row_bytes(K, w_code)], packed by
 *              bt_pack_sign (layout ROWS) from W [N, K].
 *   scale_a, scale_w  finite and > 0 (a positive scale_a leaves every sign
 *              unchanged, so it only scales the result).
 *   bias_a     device fp32 or NULL; bias_len 0, 1 or K. Ignored for BT_PACKED.
 *   out        device [M, N] in out_dtype (BT_F32, BT_BF16, BT_F16, or BT_I32
 *              for the raw dot products).
 *   algo       BT_ALGO_AUTO or the kernel matching w_code.
 *   workspace  device, >= bt_binary_linear_workspace(M, K, x_dtype, w_code)
 *              bytes, 256-byte aligned; holds the packed activations.
 * M = 0 or N = 0 is a no-op. K must be >= 1.
 */
bt_status bt_binary_linear(const void *x, bt_dtype x_dtype,
                           const void *weight, bt_code w_code,
                           int64_t M, int64_t N, int64_t K,
                           float scale_a, float scale_w,
                           const float *bias_a, int64_t bias_len,
                           void *out, bt_dtype out_dtype, bt_algo algo,
                           void *workspace, size_t workspace_bytes, bt_stream stream);

/*
 * Workspace bytes bt_binary_conv2d needs for this geometry: the packed NHWC
 * activations (unless x is packed), then, for the tensor-core codes
 * (E4M3 / E2M1), the im2col rows [B*Ho*Wo, k*k*bt_packed_row_bytes(C, code)]
 * the contraction reads, each part rounded up to 256 bytes. 0 when nothing is
 * needed (BITS with BT_PACKED x, or BT_PACKED_IM2COL x), for invalid
 * arguments, and beyond the sizes bt_binary_conv2d serves.
 */
size_t bt_binary_conv2d_workspace(int64_t B, int64_t C, int64_t H, int64_t W,
                                  int kernel_size, int stride, int padding, int dilation,
                                  bt_dtype x_dtype, bt_code code);

/*
 * bt_binary_conv2d -- BinaryConv2dForward.forward(x, weight, scale_a, scale_w,
 * is_train=False, kernel_size, stride, padding, dilation) as an im2col
 * contraction over channel-packed NHWC activations: BITS contracts the
 * packed pixels in place (the im2col is implicit, in shared memory); E4M3 /
 * E2M1 contract the weights with the im2col rows of the input (built in the
 * workspace by one fused pass over x, as bt_pack_im2col does, or unfolded
 * from packed pixels), or take those rows as BT_PACKED_IM2COL.
 *
 *   x          device NCHW [B, C, H, W] in x_dtype, or BT_PACKED:
 *              [B, H, W, bt_packed_row_bytes(C, w_code)], or BT_PACKED_IM2COL
 *              (E4M3 / E2M1 only): the rows bt_pack_im2col writes.
 *   weight     device [O, k, k, bt_packed_row_bytes(C, w_code)]: OIHW weights
 *              packed by bt_pack_sign with layout NCHW_TO_NHWC.
 *   Output size Ho = floor((H + 2p - d(k-1) - 1)/s + 1), same for Wo
 *   (banghao.live/blog/9, section 2); both must be >= 1.
 *   A tap that falls in the zero padding contributes 0 to dot (the unfold +
 *   mm lowering of that page).
 *   bias_a     device fp32 or NULL; bias_len 0, 1 or C (per input channel,
 *              bias_a.view(1,-1,1,1)). Ignored for BT_PACKED.
 *   out        device NCHW [B, O, Ho, Wo] in out_dtype.
 *   kernel_size >= 1, stride >= 1, padding >= 0, dilation >= 1.
 *   workspace  device, >= bt_binary_conv2d_workspace(B, C, H, W, kernel_size,
 *              stride, padding, dilation, x_dtype, w_code) bytes, 256-byte
 *              aligned (may be NULL when that is 0).
 * Errors: BT_ERR_WORKSPACE when the workspace is missing or too small;
 * BT_ERR_UNSUPPORTED beyond the sizes served (C*k*k > 16384 for E4M3/E2M1,
 * more than 65535*128 output pixels, H or W > 2^20).
 */
bt_status bt_binary_conv2d(const void *x, bt_dtype x_dtype,
                           const void *weight, bt_code w_code,
                           int64_t B, int64_t C, int64_t H, int64_t W, int64_t O,
                           int kernel_size, int stride, int padding, int dilation,
                           float scale_a, float scale_w,
                           const float *bias_a, int64_t bias_len,
                           void *out, bt_dtype out_dtype, bt_algo algo,
                           void *workspace, size_t workspace_bytes, bt_stream stream);

/*
 * bt_binary_linear_noalloc -- bt_binary_linear for callers that cannot
 * allocate device memory. The pages have no counterpart: it exists because
 * some callers run inside a host framework that owns every device
 * allocation (a plugin's enqueue callback, say) or under a fixed memory
 * budget, where the workspace bt_binary_linear needs cannot be obtained.
 *
 * Same arguments and result as bt_binary_linear without the workspace: the
 * packed activations go to a scratch array of
 * bt_binary_linear_noalloc_max_bytes() bytes (16 MiB) compiled into the
 * library, held in device memory of every GPU that loads it until the
 * process exits. Calls allocate nothing (no cudaMalloc / cudaFree).
 *   - A problem whose bt_binary_linear_workspace(M, K, x_dtype, w_code)
 *     exceeds that size returns BT_ERR_WORKSPACE and launches nothing.
 *   - The array's device address belongs to the CUDA context current on the
 *     calling thread: each context that loads the library (the device's
 *     primary context, a framework's own driver context) has its own copy.
 *     The first call that packs activations in a context looks that address
 *     up (cudaGetSymbolAddress, with the context current) and caches it per
 *     context; make that first call before any stream capture.
 *   - Packed activations (x_dtype BT_PACKED) and M == 0 need no scratch: such
 *     a call goes straight to bt_binary_linear with no workspace and looks
 *     nothing up.
 *   - Every call shares the one array: calls whose kernels overlap on the
 *     GPU race on it. Each call rewrites all of the scratch it reads, so
 *     nothing carries over from the previous call.
 */
bt_status bt_binary_linear_noalloc(const void *x, bt_dtype x_dtype,
                                   const void *weight, bt_code w_code,
                                   int64_t M, int64_t N, int64_t K,
                                   float scale_a, float scale_w,
                                   const float *bias_a, int64_t bias_len,
                                   void *out, bt_dtype out_dtype, bt_algo algo,
                                   bt_stream stream);

/* Size in bytes of the scratch array bt_binary_linear_noalloc uses. */
size_t bt_binary_linear_noalloc_max_bytes(void);

/*
 * bt_plan -- the "ADAPTIVE" choice: the code (weight format) and kernel this
 * build runs fastest for a problem of this size. For BT_OP_LINEAR pass
 * (M, N, K); for BT_OP_CONV2D pass M = B*Ho*Wo, N = O, K = C*k*k. A linear
 * size that bt_tune_linear has timed in this process, on the current device,
 * gets the code with the shortest measured call among those timed, and a
 * convolution size that bt_tune_conv2d has timed likewise; any other size the
 * fixed rule measured on GB300 (E2M1 up to K = 16384, else BITS).
 * Returns BT_ERR_INVALID_ARG for null outputs or sizes < 1.
 * The environment variable BT_FORCE_ALGO=popc|e4m3|e2m1 overrides it.
 */
bt_status bt_plan(bt_op op, int64_t M, int64_t N, int64_t K, bt_code *code, bt_algo *algo);

/* What bt_tune_linear measured and kept. */
typedef struct {
    bt_code code;              /* the weight's code that was timed */
    int pair;                  /* tensor-core codes: 1 = 256-row tiles on CTA pairs (cta_group::2) */
    int bn;                    /* tensor-core codes: output columns per tile */
    int slices_per_stage;      /* tensor-core codes: 128-byte K slices per pipeline stage */
    int epilogue_warps;        /* tensor-core codes: 4 or 8 */
    int candidates;            /* launch shapes timed (1 for BT_CODE_BITS) */
    float us;                  /* mean microseconds of one call in the kept shape */
    float us_model;            /* the same for the shape the cost model picks unmeasured */
} bt_tune_result;

/*
 * bt_tune_linear -- the measured form of the "ADAPTIVE" choice
 * (BinaryLinearCuda: bmm_type defaults to BMM.ADAPTIVE, which selects the
 * binary matrix-multiply kernel for the caller). Arguments as
 * bt_binary_linear (algo AUTO). For the tensor-core codes it runs the call
 * once untimed and `reps` times timed per candidate launch shape (the cost
 * model's own pick first, then the cheapest tile width by the model for every
 * other pairing and stage depth of 1 to 4 K slices, each with 4 and 8
 * epilogue warps, then narrower tiles in the model's pairing), with CUDA
 * events on `stream`, and keeps the fastest (a shape replaces the one kept so
 * far, the model's first, only when it measures more than 1 % faster, so
 * that timing noise does not move the choice): later bt_binary_linear calls on
 * this device with the same (M, N, K, w_code, out_dtype) take that shape
 * (bt_binary_linear_dscale, the first-forward and allocation-free variants
 * too). For BT_CODE_BITS it times the one kernel. Either way the time is
 * recorded against (M, N, K) for bt_plan's choice of code, so timing the same
 * size once per code (weights packed in each) lets bt_plan pick the fastest.
 * `out` holds the result of the last call. Blocks the calling thread until
 * the stream has run every timed call. reps 1..10000; result not NULL.
 * Errors: those of bt_binary_linear; BT_ERR_UNSUPPORTED while `stream` is
 * being captured into a graph. M or N zero: nothing is timed or kept.
 * The table is per process; the environment's BT_TC_CONFIG / BT_TC_EPI still
 * override it.
 */
bt_status bt_tune_linear(const void *x, bt_dtype x_dtype, const void *weight, bt_code w_code,
                         int64_t M, int64_t N, int64_t K, float scale_a, float scale_w,
                         const float *bias_a, int64_t bias_len, void *out, bt_dtype out_dtype,
                         void *workspace, size_t workspace_bytes, int reps, bt_stream stream,
                         bt_tune_result *result);

/* What bt_tune_conv2d measured and kept. */
typedef struct {
    bt_code code;              /* the weight's code that was timed */
    int pair;                  /* implicit plan: 1 = 256-channel tiles on CTA pairs (cta_group::2) */
    int weights_resident;      /* implicit plan: 1 = weights held in shared memory, 0 = streamed per tile */
    int pixel_stages;          /* implicit plan: staged pixel images in flight (1 or 2) */
    int fused;                 /* 1 = the convolution packs x itself (no NHWC pack kernel first) */
    int candidates;            /* plans timed (1 where the geometry has one route) */
    float us;                  /* mean microseconds of one call in the kept plan */
    float us_model;            /* the same for the plan the planner picks unmeasured */
    int band_split;            /* implicit plan: bands per image, as a multiple of the planner's (1, 2, 4) */
} bt_tune_conv_result;

/*
 * bt_tune_conv2d -- the measured "ADAPTIVE" choice for the convolution
 * (BinaryConv2dForward.forward runs the native convolution the layer picks).
 * Arguments as bt_binary_conv2d (algo AUTO). Where the implicit-im2col plan
 * applies (codes E4M3 / E2M1, x not BT_PACKED_IM2COL) it runs the call once
 * untimed and `reps` times timed per candidate plan -- the planner's own
 * first, then every other fitting combination of CTA pairs or single CTAs,
 * resident or streamed weights and 1 or 2 pixel stages, each also with 2 and
 * 4 times the planner's bands per image (more, narrower tiles) where that
 * changes the tiling, then each of them with the convolution packing x
 * itself where x is float and that route applies -- with CUDA events on
 * `stream`, and keeps the fastest (a plan
 * replaces the planner's only when more than 1 % faster). Later
 * bt_binary_conv2d calls on this device with the same geometry (B, C, H, W,
 * O, kernel_size, stride, padding, dilation), w_code and out_dtype take it,
 * whatever x's form; bt_conv2d_single_pass reports the kept route for the
 * geometry. Elsewhere it times the one route. Either way the time is recorded
 * against bt_plan's (M = B*Ho*Wo, N = O, K = C*k*k) for its choice of code.
 * `workspace` must hold bt_binary_conv2d_workspace(...) bytes for x's form
 * (the fused route needs none, the others what the query says). `out` holds
 * the last call's result. Blocks the calling thread until the stream has run
 * every timed call. reps 1..10000; result not NULL. Errors: those of
 * bt_binary_conv2d; BT_ERR_UNSUPPORTED while `stream` is being captured. B or
 * O zero: nothing is timed or kept. The environment's BT_CONV_PAIR /
 * BT_CONV_PLAN / BT_CONV_FUSED / BT_CONV_SPLIT still override the kept plan.
 */
bt_status bt_tune_conv2d(const void *x, bt_dtype x_dtype, const void *weight, bt_code w_code,
                         int64_t B, int64_t C, int64_t H, int64_t W, int64_t O, int kernel_size,
                         int stride, int padding, int dilation, float scale_a, float scale_w,
                         const float *bias_a, int64_t bias_len, void *out, bt_dtype out_dtype,
                         void *workspace, size_t workspace_bytes, int reps, bt_stream stream,
                         bt_tune_conv_result *result);

/* Drops every launch shape, plan and code bt_tune_linear / bt_tune_conv2d
 * kept (all devices). */
void bt_tune_reset(void);

/* The tiling of the implicit-im2col convolution (what bt_conv2d_plan_info reports). */
typedef struct {
    int implicit;           /* 1: the implicit plan applies (else the call unfolds into im2col rows) */
    int pair;               /* 1: CTA pairs, 256-channel tiles */
    int weights_resident;   /* 1: weights held in shared memory for the launch */
    int pixel_stages;       /* staged pixel images in flight (1 or 2) */
    int bands;              /* bands (tiles along the output rows) per image */
    int band_rows;          /* output rows per band */
    int cta_rows;           /* rows of a band one CTA stages (half a band for pairs) */
    int row_width;          /* virtual row width wv >= Wo: accumulator column = row * wv + column */
    int tile_n;             /* accumulator columns per tile (the MMA's N) */
    int cta_n;              /* accumulator columns per CTA (tile_n / 2 for pairs) */
    int staged_rows;        /* rows of wv pixels staged per phase image */
    int phases;             /* phase images per tile (stride 2: up to 4) */
    int max_tap_shift;      /* largest start shift, in virtual pixels, of a tap's B operand */
    int tiles;              /* tiles per launch */
    int smem_bytes;         /* dynamic shared memory per CTA */
} bt_conv_plan_info;

/*
 * bt_conv2d_plan_info -- the tiling bt_binary_conv2d's implicit-im2col
 * convolution takes for this geometry (no page counterpart: an inspection
 * call, host only, no CUDA call). code E4M3 / E2M1; out_dtype sizes the
 * epilogue's staging; sms the SMs to plan for (> 0); pair -1 for the
 * planner's choice, 0 or 1 to ask for single CTAs or pairs (pairs where they
 * fit); split >= 1 cuts each image into that many times the planner's bands
 * (BT_CONV_SPLIT). The environment's BT_CONV_* variables apply as for a
 * call. info->implicit = 0 where the implicit plan does not apply.
 * Errors: BT_ERR_INVALID_ARG (info NULL, bad sizes, code or dtype, sms < 1,
 * pair outside -1..1, split < 1).
 */
bt_status bt_conv2d_plan_info(int64_t B, int64_t C, int64_t H, int64_t W, int64_t O, int kernel_size,
                              int stride, int padding, int dilation, bt_code code, bt_dtype out_dtype,
                              int sms, int pair, int split, bt_conv_plan_info *info);

/* ------------------------------------------------------------------------
 * Device-side scales (no host synchronisation). The page's forward reads the
 * scales with .item() (BinaryConv2dForward.forward: scale_a.item() *
 * scale_w.item()), a host round trip per call; these variants take them from
 * device memory, where BinaryConv2dCutlass.set_activation's first-call
 * initialisation can be computed by bt_scale_init.
 * ------------------------------------------------------------------------ */

/*
 * bt_scale_init -- scale_out = (factor * x.abs().mean()).to(scale_dtype), the
 * activation scale BinaryConv2dCutlass.set_activation sets on the first
 * forward (factor 2 for a symmetric layer, 4 otherwise). x: n elements of
 * x_dtype (F32, BF16, F16) in device memory; the mean is the exact sum of
 * |x| (double) divided by n, rounded once to x_dtype; factor * mean is
 * rounded to x_dtype, then to scale_dtype (F32, BF16, F16); the result is
 * written as one device float. Uses one device-global accumulator per GPU:
 * calls on one GPU must not overlap. Errors: INVALID_ARG (dtypes, n < 1,
 * factor not finite > 0, null), ALIGNMENT, CUDA.
 */
bt_status bt_scale_init(const void *x, bt_dtype x_dtype, int64_t n, float factor, bt_dtype scale_dtype,
                        float *scale_out, bt_stream stream);

/*
 * bt_binary_linear_dscale / bt_binary_conv2d_dscale -- bt_binary_linear /
 * bt_binary_conv2d with the scales read on the device: `scales` points to two
 * device floats {scale_a, scale_w}, 8-byte aligned; alpha = fp32(scale_a *
 * scale_w) as for the host floats. The scales are used as they are (the host
 * cannot check them). Same results, layouts and errors otherwise.
 */
bt_status bt_binary_linear_dscale(const void *x, bt_dtype x_dtype, const void *weight, bt_code w_code, int64_t M,
                                  int64_t N, int64_t K, const float *scales, const float *bias_a, int64_t bias_len,
                                  void *out, bt_dtype out_dtype, bt_algo algo, void *workspace,
                                  size_t workspace_bytes, bt_stream stream);
bt_status bt_binary_conv2d_dscale(const void *x, bt_dtype x_dtype, const void *weight, bt_code w_code, int64_t B,
                                  int64_t C, int64_t H, int64_t W, int64_t O, int kernel_size, int stride,
                                  int padding, int dilation, const float *scales, const float *bias_a,
                                  int64_t bias_len, void *out, bt_dtype out_dtype, bt_algo algo, void *workspace,
                                  size_t workspace_bytes, bt_stream stream);

/* ------------------------------------------------------------------------
 * W8A8 im2col + gemm convolution (banghao.live/blog/9 sections 3 and 4,
 * MyQuantConv2d.forward), with optional SmoothQuant.
 * ------------------------------------------------------------------------ */

/* Workspace bytes bt_w8a8_conv2d needs (0 for invalid sizes). */
size_t bt_w8a8_conv2d_workspace(int64_t B, int64_t C, int64_t H, int64_t W, int64_t O, int kernel_size, int stride,
                                int padding, int dilation);

/*
 * bt_w8a8_conv2d -- y = (unfold(x) quantized) @ (w.view(O, -1) quantized)^T
 * reshaped to NCHW [B, O, Ho, Wo]. x NCHW and w OIHW are F32 or BF16; with
 * smooth != 0 the per-column scale s = sqrt(max|rows[:, t]| / max|w[:, t]|)
 * (fp32) divides the im2col rows and multiplies the weight first. Each side
 * is quantized per tensor: scale = fp32(max|v| / 127), q = clamp(rint(v *
 * fp32(1 / scale)), -127, 127) (torch's fake-quant rounding; q = 0 when the
 * tensor is all zeros). The integer dot products are exact (tensor cores on
 * bf16 copies of q, K split in parts of at most 1024 taps, parts added as
 * integers) and y = fp32(double(dot) * double(fp32(scale_x * scale_w))); out
 * F32 or BF16 (rounded from that fp32). k <= 8, C*k*k <= 131072 (UNSUPPORTED
 * beyond); pointers 16-byte aligned,
 * workspace 256-byte aligned (bt_w8a8_conv2d_workspace bytes); asynchronous
 * on `stream`. Errors: INVALID_ARG, ALIGNMENT, WORKSPACE, UNSUPPORTED, CUDA.
 */
bt_status bt_w8a8_conv2d(const void *x, bt_dtype x_dtype, const void *w, bt_dtype w_dtype, int64_t B, int64_t C,
                         int64_t H, int64_t W, int64_t O, int kernel_size, int stride, int padding, int dilation,
                         int smooth, void *out, bt_dtype out_dtype, void *workspace, size_t workspace_bytes,
                         bt_stream stream);

/* ------------------------------------------------------------------------
 * Backward of the binary linear layer (straight-through estimator).
 * bitorch-engine BinaryLinearForward.backward states the steps for the linear
 * layer; BinaryConv2dForward.backward writes them out (for the convolution):
 *   wt           = weight.type(grad.dtype).sign() * scale_w
 *   grad_input   = (grad @ wt) in grad's dtype, then times
 *                  middle = 1 - [x/scale_a < -1] - [x/scale_a > 1]
 *   grad_scale_a = sum(grad_input * x.sign() * (1 / sqrt(x.numel())))
 *   grad_weight  = (grad^T @ (x.sign() * scale_a)) in grad's dtype
 * The int8 quantization of grad_weight that follows on the page is left to
 * the caller. sign is torch.sign: (v > 0) - (v < 0), 0 for zeros and NaN.
 * ------------------------------------------------------------------------ */

/* Row pitch (elements) of the transposed weight signs bt_binary_linear_backward
 * takes for an N-row weight: N rounded up to 64. -1 for N < 0. */
int64_t bt_backward_weight_ld(int64_t N);

/*
 * bt_sign_transpose -- torch.sign of w, transposed, as bf16 (the
 * `weight.type(grad.dtype).sign()` of BinaryConv2dForward.backward, laid out
 * as the backward's contraction reads it). w [R, C] row-major (F32, BF16 or
 * F16); out [C, ld] bf16 with out[c*ld + r] = sign(w[r, c]) for r < R and 0
 * for R <= r < ld. Build it once per weight (like bt_pack_sign) with
 * ld = bt_backward_weight_ld(R). ld >= R and a multiple of 8; w and out
 * 16-byte aligned device memory owned by the caller.
 * Errors: INVALID_ARG (dtype, sizes, null), ALIGNMENT, UNSUPPORTED
 * (C or ld > 4,194,240), CUDA.
 */
bt_status bt_sign_transpose(const void *w, bt_dtype w_dtype, int64_t R, int64_t C, int64_t ld, void *out,
                            bt_stream stream);

/* Workspace bytes bt_binary_linear_backward needs: 0 without grad_weight;
 * else 2 * (N + K) * roundup(M, 64) bytes (each part rounded up to 256 B). */
size_t bt_binary_linear_backward_workspace(int64_t M, int64_t N, int64_t K, int want_grad_weight);

/*
 * bt_binary_linear_backward -- the gradients above for the layer
 * y = binary_linear(x, W) with upstream gradient g:
 *   x      [M, K] the forward's input, BF16 or F32 (q = x / scale_a is rounded
 *          to x's dtype before it is compared with -1 and 1);
 *   wst    [K, ldw] bf16, bt_sign_transpose(W) with ldw = bt_backward_weight_ld(N);
 *          needed only for grad_x;
 *   g      [M, N] bf16;
 *   grad_x [M, K] bf16 out (the page's fp32 grad_input holds these same
 *          values: bf16 products times 0 or 1), or NULL;
 *   grad_scale_a  one device float, overwritten with the sum (fp32 terms,
 *          summed in fp32 in no fixed order), or NULL; needs grad_x;
 *   grad_w [N, K] out, BF16 (the page's value) or F32 (the fp32 sums before
 *          the rounding to bf16), or NULL;
 *   workspace  bt_binary_linear_backward_workspace(M, N, K, grad_w != NULL)
 *          bytes, 256-byte aligned (the transposes of g and sign(x)).
 * Both products run on the tensor cores (bf16 x bf16, fp32 accumulators):
 * each output is the fp32 sum of exact products, scaled by bf16(scale) and
 * rounded once to bf16. N and K multiples of 8; scale_a, scale_w finite > 0;
 * pointers 16-byte aligned device memory owned by the caller; asynchronous on
 * `stream`. Errors: INVALID_ARG, ALIGNMENT, WORKSPACE, UNSUPPORTED (N or K
 * not a multiple of 8, no tensor-core support), CUDA.
 */
bt_status bt_binary_linear_backward(const void *x, bt_dtype x_dtype, const void *wst, int64_t ldw, const void *g,
                                    int64_t M, int64_t N, int64_t K, float scale_a, float scale_w,
                                    void *grad_x, float *grad_scale_a, void *grad_w, bt_dtype grad_w_dtype,
                                    void *workspace, size_t workspace_bytes, bt_stream stream);

/* Workspace bytes bt_binary_conv2d_backward needs for the gradients asked for
 * (0 for invalid sizes). */
size_t bt_binary_conv2d_backward_workspace(int64_t B, int64_t C, int64_t H, int64_t W, int64_t O, int kernel_size,
                                           int stride, int padding, int dilation, int want_grad_input,
                                           int want_grad_weight);

/* bt_conv2d_backward_implicit -- 1 when bt_binary_conv2d_backward computes
 * grad_x of this geometry as one implicit GEMM over the stride's sub-pixel
 * phases (O a multiple of 64, stride <= 4, kernel_size <= 8, the phases'
 * staged bands fit; BT_CONV_DGRAD=gather in the environment turns it off),
 * 0 when it takes the tap matrix and gather route. Host-side planning only:
 * touches no device. */
int bt_conv2d_backward_implicit(int64_t B, int64_t C, int64_t H, int64_t W, int64_t O, int kernel_size, int stride,
                                int padding, int dilation);

/*
 * bt_binary_conv2d_backward -- the straight-through backward of the binary
 * conv2d layer, BinaryConv2dForward.backward step by step:
 *   wt           = bf16(sign(w) * scale_w)
 *   grad_x       = bf16(conv2d_input(x.shape, wt, g)) * middle,
 *                  middle = !(q < -1 || q > 1), q = x / scale_a in x's dtype
 *   *grad_scale_a = sum(grad_x * sign(x) * fp32(1 / sqrt(B*C*H*W)))
 *   grad_w       = bf16(conv2d_weight(bf16(sign(x) * scale_a), w.shape, g))
 *   x      [B, C, H, W] NCHW, BF16 or F32;
 *   wst    [C*k*k, ldw] bf16 = bt_sign_transpose(w viewed as [O, C*k*k]),
 *          ldw = bt_backward_weight_ld(O); needed only for grad_x;
 *   g      [B, O, Ho, Wo] bf16 (Ho, Wo as in the forward);
 *   grad_x [B, C, H, W] bf16 out or NULL; grad_scale_a one device float
 *          (overwritten) or NULL, needs grad_x; grad_w [O, C, k, k] BF16 or
 *          F32 (the fp32 sums before the rounding) out, or NULL;
 *   workspace  bt_binary_conv2d_backward_workspace(...) bytes, 256-byte aligned.
 * Both gradients run on the tensor cores (bf16 operands, fp32 accumulators).
 * grad_x: where bt_conv2d_backward_implicit says so, one implicit GEMM whose
 * tiles reduce over the taps of each sub-pixel phase (the bf16 rounding, mask
 * and grad_scale_a terms in its epilogue); else a product over the unfolded
 * taps, then a gather that sums each element's taps in fp32 and rounds once.
 * grad_w: a product over the unfolded signs of x, split along the pixels and
 * summed in fp32. O a multiple of 8, B <= 65535; scales finite
 * > 0; pointers 16-byte aligned device memory owned by the caller;
 * asynchronous on `stream`. Errors: INVALID_ARG, ALIGNMENT, WORKSPACE,
 * UNSUPPORTED (O not a multiple of 8, sizes beyond the limits, no tensor
 * cores), CUDA.
 */
bt_status bt_binary_conv2d_backward(const void *x, bt_dtype x_dtype, const void *wst, int64_t ldw, const void *g,
                                    int64_t B, int64_t C, int64_t H, int64_t W, int64_t O, int kernel_size, int stride,
                                    int padding, int dilation, float scale_a, float scale_w, void *grad_x,
                                    float *grad_scale_a, void *grad_w, bt_dtype grad_w_dtype, void *workspace,
                                    size_t workspace_bytes, bt_stream stream);

/*
 * bt_binary_linear_dscale_init / bt_binary_conv2d_dscale_init -- a layer's
 * first forward, as BinaryConv2dCutlass.set_activation runs it: scale_a =
 * (factor * x.abs().mean()), the mean rounded to x's dtype, times factor
 * rounded to x's dtype, then to scale_dtype (F32, BF16, F16), is computed on
 * the device and written to scales[0]; the forward then runs with alpha =
 * fp32(scales[0] * scales[1]) (scales[1] = scale_w, read from device
 * memory). The sum of |x| comes from the same read of x that packs it: the
 * rows pack (16- or 8-byte aligned rows) and the channel-packed pixel pack
 * (16-byte aligned planes) add each thread's compensated fp32 sum of |x| (its
 * 8-element groups summed pairwise) in double, once per warp, to a
 * per-context accumulator. Where those packs do not apply, a separate pass
 * sums x in double. The sum's relative error is a few units of 2^-24; the
 * rounded scale equals (factor * exact mean) rounded as above unless the exact
 * mean lies within that error of a rounding boundary of x's dtype (for f32
 * x: within a few fp32 ulps of it). Arguments otherwise as
 * bt_binary_linear_dscale / bt_binary_conv2d_dscale with float x (the
 * workspace of bt_binary_linear_workspace / bt_binary_conv2d_workspace for
 * x's dtype); factor finite > 0. Calls on one GPU must not overlap (they
 * share the accumulator). The pages have no separate entry point: this is
 * set_activation's first call and the forward that follows, without the
 * .item() host round trip.
 */
bt_status bt_binary_linear_dscale_init(const void *x, bt_dtype x_dtype,
                                       const void *weight, bt_code w_code,
                                       int64_t M, int64_t N, int64_t K,
                                       float *scales, float factor, bt_dtype scale_dtype,
                                       const float *bias_a, int64_t bias_len,
                                       void *out, bt_dtype out_dtype, bt_algo algo,
                                       void *workspace, size_t workspace_bytes,
                                       bt_stream stream);
bt_status bt_binary_conv2d_dscale_init(const void *x, bt_dtype x_dtype,
                                       const void *weight, bt_code w_code,
                                       int64_t B, int64_t C, int64_t H, int64_t W, int64_t O,
                                       int kernel_size, int stride, int padding, int dilation,
                                       float *scales, float factor, bt_dtype scale_dtype,
                                       const float *bias_a, int64_t bias_len,
                                       void *out, bt_dtype out_dtype, bt_algo algo,
                                       void *workspace, size_t workspace_bytes,
                                       bt_stream stream);

/*
 * bt_device_status -- synchronizes `stream`, then reads and clears the
 * device error word of the current device: BT_ERR_TIMEOUT if a kernel's
 * bounded wait ran out since the last call, BT_ERR_CUDA if the stream holds a
 * CUDA error, else BT_OK.
 */
bt_status bt_device_status(bt_stream stream);

/*
 * bt_set_wait_timeout -- how long each bounded wait in the main loops of the
 * tensor-core contraction kernels (producer, MMA issuer, epilogue) waits
 * before giving up, in nanoseconds, for launches made after the call; 0
 * restores the default of 2 s. Process-wide. The pages have no counterpart:
 * it exists so that the timeout path can be exercised without breaking
 * anything -- a limit shorter than a copy's or an MMA's latency makes the
 * first real wait give up: the kernel records BT_ERR_TIMEOUT (read by
 * bt_device_status), lets its copies and MMAs in flight finish (those drains
 * always allow 2 s), frees its tensor memory and returns, and its output is
 * incomplete. Errors: INVALID_ARG for a limit above 60 s.
 */
bt_status bt_set_wait_timeout(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* BT_H */
