/*
 * CPU oracle for the binarized linear / conv2d forward.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library links, includes or calls
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark load it. It shares no code, header, table or constant with the
 * CUDA path.
 *
 * What it computes is the plain definition, written out as nested loops over
 * unpacked +1/-1 int8 arrays (no bit packing, no popcount, no blocking):
 *
 *   binarize   s = +1 if (x + bias) >= 0 else -1, the sum taken in double.
 *              bitorch-engine, BinaryConv2dCutlass.set_activation (the
 *              "learnable shift input" x + bias_a.view(1,-1,1,1)); the
 *              threshold at zero and the +1 for a zero are the plain reading
 *              of "sign binarization" with value >= 0 -> +1.
 *   linear     dot[m,n] = sum_k sa[m,k] * sw[n,k]   (i-j-k loop, the shape of
 *              LinearAPoT.matmul on the torch/ao/quantization/experimental
 *              linear.py page), the contraction that BinaryLinearForward
 *              .forward scales by scale_a * scale_w.
 *   conv2d     dot[b,o,i,j] = sum_c sum_kh sum_kw [tap inside the image]
 *                             * sa[b,c,y,x] * sw[o,c,kh,kw],
 *              y = i*s - p + kh*d, x = j*s - p + kw*d, with the output size
 *              h_out = floor((h + 2p - d(k-1) - 1)/s + 1) of the im2col+gemm
 *              page (banghao.live/blog/9, section 2, MyConv2d.forward).
 *              A tap that falls in the zero padding contributes 0, exactly as
 *              in that page's unfold (zero padded) + mm lowering.
 *
 * Integer results are exact: |dot| <= K < 2^31.
 */
#include <stdint.h>
#include <stddef.h>

/* s[i] = +1 if (double)x[i] + (double)bias >= 0 else -1.
 * bias_len == 0: no bias. Otherwise element i uses bias[(i / inner) % bias_len]
 * (a scalar: bias_len = 1; per channel of NCHW: inner = H*W, bias_len = C;
 * per feature of a row-major [R,K] matrix: inner = 1, bias_len = K).
 * A NaN input compares false and gives -1. */
void orc_binarize(const float *x, int64_t n, const float *bias, int64_t bias_len,
                  int64_t inner, int8_t *s)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double b = 0.0;
        if (bias_len > 0)
            b = (double)bias[(i / inner) % bias_len];
        double v = (double)x[i] + b;
        s[i] = (v >= 0.0) ? (int8_t)1 : (int8_t)-1;
    }
}

/* dot[m*N + n] = sum_{k<K} sa[m*K + k] * sw[n*K + k] */
void orc_linear_dot(const int8_t *sa, const int8_t *sw, int64_t M, int64_t N, int64_t K,
                    int32_t *dot)
{
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            int32_t acc = 0;
            for (int64_t k = 0; k < K; ++k)
                acc += (int32_t)sa[m * K + k] * (int32_t)sw[n * K + k];
            dot[m * N + n] = acc;
        }
    }
}

/* The same sum for a list of (row, col) pairs only. */
void orc_linear_dot_at(const int8_t *sa, const int8_t *sw, int64_t K,
                       const int64_t *rows, const int64_t *cols, int64_t count, int32_t *dot)
{
    #pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < count; ++t) {
        int64_t m = rows[t], n = cols[t];
        int32_t acc = 0;
        for (int64_t k = 0; k < K; ++k)
            acc += (int32_t)sa[m * K + k] * (int32_t)sw[n * K + k];
        dot[t] = acc;
    }
}

static int64_t out_size(int64_t h, int64_t k, int64_t s, int64_t p, int64_t d)
{
    /* floor((h + 2p - d(k-1) - 1)/s + 1); the numerator may be negative, in
     * which case there is no output (the caller rejects that shape). */
    int64_t num = h + 2 * p - d * (k - 1) - 1;
    if (num < 0)
        return 0;
    return num / s + 1;
}

/* One output element of the direct convolution. sa is NCHW [B,C,H,W] and
 * sw is OIHW [O,C,k,k], both +1/-1. */
static int32_t conv_point(const int8_t *sa, const int8_t *sw, int64_t C, int64_t H, int64_t W,
                          int64_t k, int64_t s, int64_t p, int64_t d,
                          int64_t b, int64_t o, int64_t i, int64_t j)
{
    int32_t acc = 0;
    for (int64_t c = 0; c < C; ++c) {
        for (int64_t kh = 0; kh < k; ++kh) {
            for (int64_t kw = 0; kw < k; ++kw) {
                int64_t y = i * s - p + kh * d;
                int64_t x = j * s - p + kw * d;
                if (y < 0 || y >= H || x < 0 || x >= W)
                    continue; /* zero padding: contributes 0 */
                int32_t a = sa[((b * C + c) * H + y) * W + x];
                int32_t w = sw[((o * C + c) * k + kh) * k + kw];
                acc += a * w;
            }
        }
    }
    return acc;
}

/* dot is NCHW [B,O,Ho,Wo]. */
void orc_conv2d_dot(const int8_t *sa, const int8_t *sw, int64_t B, int64_t C, int64_t H,
                    int64_t W, int64_t O, int64_t k, int64_t s, int64_t p, int64_t d,
                    int32_t *dot)
{
    int64_t Ho = out_size(H, k, s, p, d);
    int64_t Wo = out_size(W, k, s, p, d);
    #pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t b = 0; b < B; ++b)
        for (int64_t o = 0; o < O; ++o)
            for (int64_t i = 0; i < Ho; ++i)
                for (int64_t j = 0; j < Wo; ++j)
                    dot[((b * O + o) * Ho + i) * Wo + j] =
                        conv_point(sa, sw, C, H, W, k, s, p, d, b, o, i, j);
}

/* The same for a list of flat NCHW output indices only. */
void orc_conv2d_dot_at(const int8_t *sa, const int8_t *sw, int64_t B, int64_t C, int64_t H,
                       int64_t W, int64_t O, int64_t k, int64_t s, int64_t p, int64_t d,
                       const int64_t *index, int64_t count, int32_t *dot)
{
    int64_t Ho = out_size(H, k, s, p, d);
    int64_t Wo = out_size(W, k, s, p, d);
    (void)B;
    #pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < count; ++t) {
        int64_t r = index[t];
        int64_t j = r % Wo; r /= Wo;
        int64_t i = r % Ho; r /= Ho;
        int64_t o = r % O;  r /= O;
        int64_t b = r;
        dot[t] = conv_point(sa, sw, C, H, W, k, s, p, d, b, o, i, j);
    }
}

int64_t orc_conv2d_out_size(int64_t h, int64_t k, int64_t s, int64_t p, int64_t d)
{
    return out_size(h, k, s, p, d);
}
