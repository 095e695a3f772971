"""Pins for the CPU oracle, checked against things other than itself.

Each pin comes from the sources (bitorch-engine's binary layers, the
im2col+gemm write-up) or from mathematics: hand-worked examples
(tests/golden/hand_examples.json), brute force with Python integers on tiny
inputs, the invariants of a +1/-1 dot product (|dot| <= K, dot = K (mod 2),
dot = K - 2*hamming), torch's own conv2d and the unfold + mm lowering of
banghao.live/blog/9 section 2, the output-size formula of that section, and
exact IEEE rounding cases worked out by hand. The last tests plant plausible
mistakes in copies of the oracle's arithmetic and check that these pins
catch them.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


def _rand_pm1(rng, shape):
    return np.where(rng.random(shape) < 0.5, 1, -1).astype(np.int8)


# ---------------------------------------------------------------------------
# Hand-worked examples
# ---------------------------------------------------------------------------

def test_golden_linear():
    for ex in json.load(open(GOLDEN))["linear"]:
        x = torch.tensor(ex["x"], dtype=torch.float32)
        w = torch.tensor(ex["w"], dtype=torch.float32)
        bias = torch.tensor(ex["bias"]) if "bias" in ex else None
        sa = oracle.binarize(x, bias, channel_axis=-1)
        sw = oracle.binarize_weight(w)
        np.testing.assert_array_equal(oracle.linear_dot(sa, sw), np.array(ex["dot"]), ex["why"])


def test_golden_conv():
    for ex in json.load(open(GOLDEN))["conv"]:
        sa = oracle.binarize(torch.tensor(ex["x"]))
        sw = oracle.binarize_weight(torch.tensor(ex["w"]))
        got = oracle.conv2d_dot(sa, sw, ex["stride"], ex["padding"], ex["dilation"])
        np.testing.assert_array_equal(got, np.array(ex["dot"]), ex["why"])


def test_golden_pack():
    g = json.load(open(GOLDEN))
    for ex in g["pack_bits"]:
        if "signs" in ex:
            s = np.array([ex["signs"]], np.int8)
        elif "signs_all_plus" in ex:
            s = np.ones((1, ex["signs_all_plus"]), np.int8)
        else:
            s = np.array([[-1] * ex["signs_neg_then_plus"] + [1]], np.int8)
        words = oracle.pack_rows(s, oracle.CODE_BITS).view(np.uint32)[0]
        np.testing.assert_array_equal(words, np.array(ex["words"], np.uint32), ex["why"])
    for ex in g["pack_codes"]:
        code = {"e4m3": oracle.CODE_E4M3, "e2m1": oracle.CODE_E2M1}[ex["code"]]
        got = oracle.pack_rows(np.array([ex["signs"]], np.int8), code)[0]
        n = len(ex["bytes"])
        assert got.size == 64
        np.testing.assert_array_equal(got[:n], np.array(ex["bytes"], np.uint8), ex["why"])
        assert not got[n:].any()


def test_code_values_decode_to_plus_minus_one():
    # E4M3 through torch's own float8 type.
    b = torch.tensor([0x38, 0xB8, 0x00], dtype=torch.uint8)
    np.testing.assert_array_equal(b.view(torch.float8_e4m3fn).float().numpy(), [1.0, -1.0, 0.0])

    # E2M1 by its definition: sign bit 3, exponent bits 2..1 with bias 1, mantissa bit 0.
    def e2m1(n):
        sign = -1.0 if n & 0x8 else 1.0
        e, m = (n >> 1) & 0x3, n & 0x1
        return sign * (m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + 0.5 * m))

    assert (e2m1(0x2), e2m1(0xA), e2m1(0x0)) == (1.0, -1.0, 0.0)


# ---------------------------------------------------------------------------
# Binarization rule
# ---------------------------------------------------------------------------

def test_binarize_special_values():
    tiny = np.float32(1e-45)          # smallest positive subnormal
    cases = [
        (0.0, None, 1), (-0.0, None, 1), (tiny, None, 1), (-tiny, None, -1),
        (np.nan, None, -1), (np.inf, None, 1), (-np.inf, None, -1),
        (0.5, -0.5, 1),                                   # x == -bias exactly: sum is 0
        (0.5, -np.nextafter(np.float32(0.5), np.float32(1)), -1),  # sum is -2^-24
        (-1e-40, 0.0, -1), (1e-40, -1e-40, 1),            # subnormals, no flush to zero
        (3.0, -np.inf, -1), (np.inf, -np.inf, -1),        # inf - inf is NaN -> -1
        (1.0e30, -1.0e30, 1), (-3.0, 2.5, -1),
    ]
    for x, b, want in cases:
        bias = None if b is None else np.array([b], np.float32)
        got = oracle.binarize(np.array([x], np.float32), bias)[0]
        assert got == want, (x, b)


def test_binarize_bf16_and_f16_inputs_are_exact():
    v = torch.tensor([-1.0e-38, 1.0e-38, -0.0, 3.5, -3.5])
    for dt in (torch.bfloat16, torch.float16):
        got = oracle.binarize(v.to(dt))
        want = [(-1 if float(t) < 0 else 1) for t in v.to(dt).float()]
        np.testing.assert_array_equal(got, want)


def test_binarize_per_channel_bias_uses_channel_axis():
    x = torch.zeros(2, 3, 2, 2)
    bias = torch.tensor([-1.0, 0.0, 1.0])
    s = oracle.binarize(x, bias, channel_axis=1)
    assert (s[:, 0] == -1).all() and (s[:, 1] == 1).all() and (s[:, 2] == 1).all()
    x2 = torch.full((2, 3), 0.5)
    s2 = oracle.binarize(x2, torch.tensor([-1.0, -0.5, 0.0]), channel_axis=-1)
    np.testing.assert_array_equal(s2, [[-1, 1, 1], [-1, 1, 1]])


# ---------------------------------------------------------------------------
# Linear: brute force, invariants, special cases
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("K", [1, 31, 32, 33, 63, 64, 65, 127, 4100])
def test_linear_brute_force(K):
    rng = np.random.default_rng(K)
    M, N = (3, 4) if K > 1000 else (5, 7)
    sa, sw = _rand_pm1(rng, (M, K)), _rand_pm1(rng, (N, K))
    got = oracle.linear_dot(sa, sw)
    a, w = sa.tolist(), sw.tolist()
    for m in range(M):
        for n in range(N):
            assert got[m, n] == sum(a[m][k] * w[n][k] for k in range(K))


@pytest.mark.parametrize("K", [7, 64, 300, 1031])
def test_linear_invariants(K):
    rng = np.random.default_rng(100 + K)
    sa, sw = _rand_pm1(rng, (9, K)), _rand_pm1(rng, (11, K))
    dot = oracle.linear_dot(sa, sw).astype(np.int64)
    ham = np.array([[np.count_nonzero((sa[m] > 0) != (sw[n] > 0)) for n in range(11)]
                    for m in range(9)])
    np.testing.assert_array_equal(dot, K - 2 * ham)
    assert (np.abs(dot) <= K).all()
    assert ((dot - K) % 2 == 0).all()


def test_linear_special_cases():
    rng = np.random.default_rng(7)
    K = 257
    w = _rand_pm1(rng, (6, K))
    np.testing.assert_array_equal(np.diag(oracle.linear_dot(w, w)), [K] * 6)
    np.testing.assert_array_equal(np.diag(oracle.linear_dot(-w, w)), [-K] * 6)
    ones = np.ones((1, K), np.int8)
    np.testing.assert_array_equal(oracle.linear_dot(ones, w)[0], w.astype(np.int64).sum(1))


def test_linear_matches_float64_matmul_of_signs():
    rng = np.random.default_rng(3)
    x = torch.from_numpy(rng.standard_normal((33, 517)).astype(np.float32))
    w = torch.from_numpy(rng.standard_normal((19, 517)).astype(np.float32))
    sx = torch.where(x >= 0, 1.0, -1.0).double()
    sw = torch.where(w >= 0, 1.0, -1.0).double()
    want = (sx @ sw.T).numpy()
    got = oracle.linear_dot(oracle.binarize(x), oracle.binarize_weight(w))
    np.testing.assert_array_equal(got, want)


def test_linear_dot_at_agrees_with_full():
    rng = np.random.default_rng(11)
    sa, sw = _rand_pm1(rng, (40, 77)), _rand_pm1(rng, (30, 77))
    full = oracle.linear_dot(sa, sw)
    rows, cols = rng.integers(0, 40, 50), rng.integers(0, 30, 50)
    np.testing.assert_array_equal(oracle.linear_dot_at(sa, sw, rows, cols), full[rows, cols])


# ---------------------------------------------------------------------------
# Conv: output size, torch conv2d, unfold + mm, brute force, invariants
# ---------------------------------------------------------------------------

CONV_GRID = [
    # (B, C, H, W, O, k, s, p, d)
    (1, 1, 5, 5, 1, 3, 1, 1, 1), (2, 3, 7, 6, 4, 3, 2, 1, 1), (1, 31, 6, 6, 3, 1, 1, 0, 1),
    (2, 33, 5, 7, 2, 3, 1, 2, 2), (1, 64, 9, 9, 5, 5, 3, 3, 1), (1, 4, 1, 1, 2, 3, 1, 1, 1),
    (1, 2, 8, 8, 3, 3, 2, 2, 2), (3, 5, 4, 9, 2, 5, 1, 2, 1), (1, 3, 11, 11, 2, 3, 3, 0, 2),
]


@pytest.mark.parametrize("B,C,H,W,O,k,s,p,d", CONV_GRID)
def test_conv_matches_torch_conv2d(B, C, H, W, O, k, s, p, d):
    rng = np.random.default_rng(B * 1000 + C * 10 + k)
    sa, sw = _rand_pm1(rng, (B, C, H, W)), _rand_pm1(rng, (O, C, k, k))
    want = F.conv2d(torch.from_numpy(sa).double(), torch.from_numpy(sw).double(),
                    stride=s, padding=p, dilation=d)
    got = oracle.conv2d_dot(sa, sw, s, p, d)
    assert got.shape == tuple(want.shape)
    np.testing.assert_array_equal(got, want.numpy())


@pytest.mark.parametrize("B,C,H,W,O,k,s,p,d", CONV_GRID)
def test_conv_matches_unfold_mm(B, C, H, W, O, k, s, p, d):
    # banghao.live/blog/9 section 2: unfold -> [bs*L, C*k*k] -> mm(W.view(O,-1).T)
    # -> reshape to [bs, O, h_out, w_out]; dilation is passed to unfold here.
    rng = np.random.default_rng(7 + C + H)
    sa, sw = _rand_pm1(rng, (B, C, H, W)), _rand_pm1(rng, (O, C, k, k))
    ho = (H + 2 * p - d * (k - 1) - 1) // s + 1
    wo = (W + 2 * p - d * (k - 1) - 1) // s + 1
    cols = F.unfold(torch.from_numpy(sa).double(), kernel_size=k, padding=p, stride=s, dilation=d)
    L = cols.shape[2]
    cols = cols.transpose(1, 2).reshape(-1, C * k * k)
    out = torch.mm(cols, torch.from_numpy(sw).double().view(O, -1).t())
    out = out.reshape(B, L, O).transpose(1, 2).reshape(B, O, ho, wo)
    np.testing.assert_array_equal(oracle.conv2d_dot(sa, sw, s, p, d), out.numpy())


def test_conv_output_size_formula():
    for h, k, s, p, d in itertools.product([1, 5, 14, 28], [1, 3, 5], [1, 2, 3], [0, 1, 2], [1, 2]):
        num = h + 2 * p - d * (k - 1) - 1
        got = oracle.conv2d_out_size(h, k, s, p, d)
        if num < 0:
            assert got == 0
            continue
        ref = F.conv2d(torch.zeros(1, 1, h, h), torch.zeros(1, 1, k, k), stride=s, padding=p,
                       dilation=d).shape[-1]
        assert got == ref


def test_conv_brute_force_python_loops():
    rng = np.random.default_rng(5)
    B, C, H, W, O, k, s, p, d = 2, 2, 4, 5, 2, 3, 2, 2, 2
    sa, sw = _rand_pm1(rng, (B, C, H, W)), _rand_pm1(rng, (O, C, k, k))
    got = oracle.conv2d_dot(sa, sw, s, p, d)
    ho, wo = got.shape[2:]
    for b, o, i, j in itertools.product(range(B), range(O), range(ho), range(wo)):
        acc = 0
        for c, kh, kw in itertools.product(range(C), range(k), range(k)):
            y, x = i * s - p + kh * d, j * s - p + kw * d
            if 0 <= y < H and 0 <= x < W:
                acc += int(sa[b, c, y, x]) * int(sw[o, c, kh, kw])
        assert got[b, o, i, j] == acc


def test_conv_invariants_with_valid_tap_count():
    rng = np.random.default_rng(9)
    B, C, H, W, O, k, s, p, d = 2, 5, 6, 6, 3, 3, 1, 2, 1
    sa, sw = _rand_pm1(rng, (B, C, H, W)), _rand_pm1(rng, (O, C, k, k))
    dot = oracle.conv2d_dot(sa, sw, s, p, d).astype(np.int64)
    ho, wo = dot.shape[2:]
    for i, j in itertools.product(range(ho), range(wo)):
        nv = sum(1 for kh in range(k) for kw in range(k)
                 if 0 <= i * s - p + kh * d < H and 0 <= j * s - p + kw * d < W)
        assert (np.abs(dot[:, :, i, j]) <= C * nv).all()
        assert ((dot[:, :, i, j] - C * nv) % 2 == 0).all()


def test_conv_dot_at_agrees_with_full():
    rng = np.random.default_rng(21)
    sa, sw = _rand_pm1(rng, (2, 6, 7, 7)), _rand_pm1(rng, (4, 6, 3, 3))
    full = oracle.conv2d_dot(sa, sw, 2, 1, 1)
    idx = rng.integers(0, full.size, 64)
    np.testing.assert_array_equal(oracle.conv2d_dot_at(sa, sw, 2, 1, 1, idx), full.reshape(-1)[idx])


def test_pack_nhwc_is_channel_rows():
    rng = np.random.default_rng(4)
    s = _rand_pm1(rng, (2, 37, 3, 4))
    for code in (oracle.CODE_BITS, oracle.CODE_E4M3, oracle.CODE_E2M1):
        p = oracle.pack_nchw_to_nhwc(s, code)
        assert p.shape == (2, 3, 4, oracle.packed_row_bytes(37, code))
        np.testing.assert_array_equal(p[1, 2, 3], oracle.pack_rows(s[1, :, 2, 3][None], code)[0])


# ---------------------------------------------------------------------------
# Epilogue: exact rounding cases worked by hand
# ---------------------------------------------------------------------------

def test_alpha_rounds_the_exact_product_once_to_float():
    # (1 + 2^-12)^2 = 1 + 2^-11 + 2^-24: the 2^-24 term is half an ulp of 1.0
    # in fp32, a tie, rounded to the even neighbour 1 + 2^-11.
    a = 1.0 + 2.0 ** -12
    assert oracle.alpha(a, a) == np.float32(1.0 + 2.0 ** -11)
    # (1 + 2^-12)(1 + 2^-11) = 1 + 3*2^-12 + 2^-23: exactly representable.
    assert oracle.alpha(a, 1.0 + 2.0 ** -11) == np.float32(1.0 + 3 * 2.0 ** -12 + 2.0 ** -23)


def test_epilogue_bf16_round_half_even():
    dot = np.array([1, 1, -1, 2], np.int32)
    # 1 + 2^-8 sits halfway between bf16 neighbours 1 and 1 + 2^-7 -> even (1.0)
    y = oracle.epilogue(dot[:1], 1.0 + 2.0 ** -8, 1.0, "bf16")
    assert y.dtype == torch.bfloat16 and float(y[0]) == 1.0
    # 1 + 3*2^-8 sits halfway between 1 + 2^-7 and 1 + 2^-6 -> even (1 + 2^-6)
    y = oracle.epilogue(dot, 1.0 + 3 * 2.0 ** -8, 1.0, "bf16")
    assert [float(v) for v in y] == [1.015625, 1.015625, -1.015625, 2.03125]
    # just above the tie rounds up
    y = oracle.epilogue(dot[:1], 1.0 + 2.0 ** -8 + 2.0 ** -20, 1.0, "bf16")
    assert float(y[0]) == 1.0 + 2.0 ** -7


def test_epilogue_f32_and_i32():
    dot = np.array([0, 3, -11008, 4096], np.int32)
    a = 1.0 + 2.0 ** -12
    y = oracle.epilogue(dot, a, a, "f32")
    al = 1.0 + 2.0 ** -11
    assert y.dtype == torch.float32
    assert [float(v) for v in y] == [0.0, 3 * al, -11008 * al, 4096 * al]
    np.testing.assert_array_equal(oracle.epilogue(dot, a, a, "i32").numpy(), dot)


def test_epilogue_f32_single_rounding_of_product():
    # dot = 3, alpha = 1 + 2^-23 (one ulp above 1): 3 + 3*2^-23 = 3 + 1.5 ulp
    # (the ulp in [2,4) is 2^-22), a tie between 3 + 2^-22 (odd last bit) and
    # 3 + 2^-21 (even) -> 3 + 2^-21. dot = 5: the ulp in [4,8) is 2^-21, so
    # 5 + 5*2^-23 = 5 + 1.25 ulp -> 5 + 2^-21.
    y = oracle.epilogue(np.array([3, 5], np.int32), 1.0 + 2.0 ** -23, 1.0, "f32")
    assert float(y[0]) == 3.0 + 2.0 ** -21
    assert float(y[1]) == 5.0 + 2.0 ** -21


# ---------------------------------------------------------------------------
# Whole forward composed from the parts, and the workload recipe
# ---------------------------------------------------------------------------

def test_binary_linear_composition():
    wl = workloads.tiny_linear()
    y = oracle.binary_linear(wl.x, wl.w, wl.scale_a, wl.scale_w, wl.bias, wl.out_dtype)
    sx = torch.where(wl.x >= 0, 1.0, -1.0).double()
    sw = torch.where(wl.w >= 0, 1.0, -1.0).double()
    ref = (sx @ sw.T) * float(np.float32(np.float64(wl.scale_a) * np.float64(wl.scale_w)))
    assert y.shape == (64, 256) and y.dtype == torch.float32
    torch.testing.assert_close(y.double(), ref, rtol=1e-7, atol=0)


def test_workload_recipe():
    wl = workloads.tiny_linear()
    assert tuple(wl.x.shape) == (64, 512) and tuple(wl.w.shape) == (256, 512)
    assert wl.bias is None and wl.out_dtype == "f32"
    assert wl.scale_a == pytest.approx(float(wl.x.abs().double().mean()), rel=1e-7)
    again = workloads.tiny_linear()
    assert torch.equal(wl.x, again.x) and torch.equal(wl.w, again.w)
    assert wl.gemm_shape() == (64, 256, 512)
    c = workloads.conv("c", 2, 3, 14, 14, 4, 3, 2, 1, 1)
    assert c.gemm_shape() == (2 * 7 * 7, 4, 27)


# ---------------------------------------------------------------------------
# Planted mistakes: plausible errors in copies of the oracle's arithmetic
# must fail the pins above.
# ---------------------------------------------------------------------------

def _conv_mutant(sa, sw, s, p, d, mistake):
    B, C, H, W = sa.shape
    O, _, k, _ = sw.shape
    ho, wo = (H + 2 * p - d * (k - 1) - 1) // s + 1, (W + 2 * p - d * (k - 1) - 1) // s + 1
    out = np.zeros((B, O, ho, wo), np.int64)
    for b, o, i, j in itertools.product(range(B), range(O), range(ho), range(wo)):
        for c, kh, kw in itertools.product(range(C), range(k), range(k)):
            y, x = i * s - p + kh * d, j * s - p + kw * d
            if mistake == "flipped_kernel":
                wv = sw[o, c, k - 1 - kh, k - 1 - kw]
            elif mistake == "swapped_taps":
                wv = sw[o, c, kw, kh]
            else:
                wv = sw[o, c, kh, kw]
            if mistake == "no_dilation":
                y, x = i * s - p + kh, j * s - p + kw
            if 0 <= y < H and 0 <= x < W:
                out[b, o, i, j] += int(sa[b, c, y, x]) * int(wv)
            elif mistake == "pad_as_plus_one":
                out[b, o, i, j] += int(wv)
    return out


@pytest.mark.parametrize("mistake", ["flipped_kernel", "swapped_taps", "no_dilation",
                                     "pad_as_plus_one"])
def test_planted_conv_mistakes_are_caught(mistake):
    rng = np.random.default_rng(31)
    sa, sw = _rand_pm1(rng, (1, 3, 6, 6)), _rand_pm1(rng, (2, 3, 3, 3))
    want = F.conv2d(torch.from_numpy(sa).double(), torch.from_numpy(sw).double(),
                    stride=1, padding=2, dilation=2).numpy()
    assert np.array_equal(_conv_mutant(sa, sw, 1, 2, 2, None), want)
    assert not np.array_equal(_conv_mutant(sa, sw, 1, 2, 2, mistake), want)


def test_planted_linear_mistakes_are_caught():
    rng = np.random.default_rng(32)
    K = 33
    sa, sw = _rand_pm1(rng, (4, K)), _rand_pm1(rng, (5, K))
    ham = np.array([[np.count_nonzero((sa[m] > 0) != (sw[n] > 0)) for n in range(5)]
                    for m in range(4)])
    good = sa.astype(np.int64) @ sw.T.astype(np.int64)
    assert np.array_equal(good, K - 2 * ham)
    dropped_last = sa[:, :-1].astype(np.int64) @ sw[:, :-1].T.astype(np.int64)
    assert not np.array_equal(dropped_last, K - 2 * ham)
    wrong_sign = -good
    assert not np.array_equal(wrong_sign, K - 2 * ham)
    # a threshold of > 0 instead of >= 0 changes the sign of exact zeros
    x = np.array([[0.0, 1.0, -1.0]], np.float32)
    assert oracle.binarize(x)[0, 0] == 1 and np.where(x > 0, 1, -1)[0, 0] == -1


# ---------------------------------------------------------------------------
# Backward of the binary linear layer (straight-through estimator)
# ---------------------------------------------------------------------------

def test_golden_linear_backward():
    for ex in json.load(open(GOLDEN))["linear_backward"]:
        got = oracle.linear_backward(np.array(ex["x"], np.float32), np.array(ex["w"], np.float32),
                                     np.array(ex["g"], np.float32), ex["scale_a"], ex["scale_w"], ex["x_dtype"])
        np.testing.assert_array_equal(got["grad_input"], np.array(ex["grad_input"], np.float32), ex["why"])
        np.testing.assert_array_equal(got["grad_weight"], np.array(ex["grad_weight"], np.float32), ex["why"])
        assert got["grad_scale_a"] == ex["grad_scale_a"], ex["why"]
        if "grad_input_if_f32_x" in ex:
            got32 = oracle.linear_backward(np.array(ex["x"], np.float32), np.array(ex["w"], np.float32),
                                           np.array(ex["g"], np.float32), ex["scale_a"], ex["scale_w"], "f32")
            np.testing.assert_array_equal(got32["grad_input"], np.array(ex["grad_input_if_f32_x"], np.float32))


def test_sign_matches_torch_sign():
    v = np.array([-0.0, 0.0, np.nan, -np.nan, 2.0, -3.0, 1e-45, -1e-45, np.inf, -np.inf], np.float32)
    want = torch.from_numpy(v).sign().numpy()
    got = oracle.sign(v)
    np.testing.assert_array_equal(got, want)
    assert not np.signbit(got[0]) and not np.isnan(got[2])


def test_bf16_round_matches_torch_cast():
    rng = np.random.default_rng(41)
    v = np.concatenate([rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 20000),
                        np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 3.39e38, 3.4e38, 1e-39, -1e-41,
                                  2.0 ** -133, 1.5 * 2.0 ** -133, 2.5 * 2.0 ** -133], np.float32)]).astype(np.float32)
    # exact ties: 1 + (2j + 1) * 2^-8 sit halfway between bf16 neighbours
    ties = (1.0 + (2 * np.arange(64) + 1) * 2.0 ** -8).astype(np.float32)
    v = np.concatenate([v, ties, -ties])
    want = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    got = oracle.bf16_round(v)
    np.testing.assert_array_equal(got, want)
    num = ~np.isnan(want)
    assert np.array_equal(np.signbit(got[num]), np.signbit(want[num]))


def _ste_autograd(x, w, g, scale_a, scale_w, x_dtype):
    """The straight-through gradients by torch autograd in float64: the
    activation passes through a clamp-like function whose derivative is 1
    where |x / scale_a| < 1 and 0 outside; the weight enters as sign(w)
    rounded to bf16 times scale_w, with an identity derivative for w."""
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    wt = torch.tensor(w, dtype=torch.float64, requires_grad=True)
    s_w = torch.from_numpy(oracle.bf16_round(torch.from_numpy(np.asarray(w, np.float32)).sign().numpy() * np.float32(scale_w))).double()
    s_x = torch.from_numpy(oracle.bf16_round(torch.from_numpy(np.asarray(x, np.float32)).sign().numpy() * np.float32(scale_a))).double()
    act = torch.nn.functional.hardtanh(xt / scale_a) * scale_a        # derivative: 1 strictly inside
    wq = s_w + (wt - wt.detach())                                       # value s_w, derivative 1
    y = act @ s_w.T + s_x @ wq.T - s_x @ s_w.T.detach()                 # splits the two paths
    (y * torch.tensor(g, dtype=torch.float64)).sum().backward()
    return xt.grad.numpy(), wt.grad.numpy()


@pytest.mark.parametrize("M,N,K", [(3, 4, 5), (8, 16, 7), (1, 33, 64)])
def test_linear_backward_matches_autograd(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    scale_a, scale_w = 0.75, 0.3
    x = torch.randn(M, K, generator=torch.Generator().manual_seed(K)).to(torch.bfloat16).float().numpy()
    # keep |x / scale_a| away from 1, where bf16 rounding of the quotient decides the mask
    r = np.abs(x / scale_a)
    x[(r > 1 - 2.0 ** -6) & (r < 1 + 2.0 ** -6)] = 0.0
    w = rng.standard_normal((N, K)).astype(np.float32)
    w[0, 0] = 0.0                                                       # sign(0) = 0
    g = torch.randn(M, N, generator=torch.Generator().manual_seed(N)).to(torch.bfloat16).float().numpy()
    o = oracle.linear_backward(x, w, g, scale_a, scale_w, "bf16")
    gx, gw = _ste_autograd(x, w, g, scale_a, scale_w, "bf16")
    np.testing.assert_allclose(o["grad_input_exact"] * o["middle"], gx, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o["grad_weight_exact"], gw, rtol=0, atol=1e-12)


def test_linear_backward_closed_forms():
    rng = np.random.default_rng(43)
    M, N, K = 5, 7, 9
    scale_a, scale_w = 0.6, 0.45
    x = (np.abs(torch.randn(M, K).to(torch.bfloat16).float().numpy()) * 0.5).astype(np.float32) + 0.01
    g = torch.randn(M, N).to(torch.bfloat16).float().numpy()
    w = np.abs(rng.standard_normal((N, K))).astype(np.float32) + 0.1   # every sign +1
    o = oracle.linear_backward(x, w, g, scale_a, scale_w, "bf16")
    bw = np.float64(oracle.bf16_round(np.float32(scale_w)))
    ba = np.float64(oracle.bf16_round(np.float32(scale_a)))
    # all weights +1: every grad_input column is bf16(scale_w) times the row sum of g
    np.testing.assert_array_equal(o["grad_input_exact"], np.repeat(bw * g.astype(np.float64).sum(1, keepdims=True), K, 1))
    # all activations positive: every grad_weight column is bf16(scale_a) times the column sum of g
    np.testing.assert_array_equal(o["grad_weight_exact"], np.repeat(ba * g.astype(np.float64).sum(0)[:, None], K, 1))
    # doubling g doubles every gradient exactly (power-of-two scaling commutes with rounding)
    o2 = oracle.linear_backward(x, w, 2 * g, scale_a, scale_w, "bf16")
    np.testing.assert_array_equal(o2["grad_input"], 2 * o["grad_input"])
    np.testing.assert_array_equal(o2["grad_weight"], 2 * o["grad_weight"])
    assert o2["grad_scale_a"] == 2 * o["grad_scale_a"]
    # outside |x| <= scale_a the input gradient is zero
    x[0, 0] = 3.0
    o3 = oracle.linear_backward(x, w, g, scale_a, scale_w, "bf16")
    assert o3["middle"][0, 0] == 0 and o3["grad_input"][0, 0] == 0


def test_planted_backward_mistakes_are_caught():
    rng = np.random.default_rng(44)
    M, N, K = 4, 6, 5
    x = torch.randn(M, K, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).float().numpy()
    x[np.abs(np.abs(x / 0.8) - 1) < 2.0 ** -6] = 0.0
    w = rng.standard_normal((N, K)).astype(np.float32)
    g = torch.randn(M, N, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16).float().numpy()
    gx, gw = _ste_autograd(x, w, g, 0.8, 0.3, "bf16")
    o = oracle.linear_backward(x, w, g, 0.8, 0.3, "bf16")
    assert np.allclose(o["grad_input_exact"] * o["middle"], gx) and np.allclose(o["grad_weight_exact"], gw)
    wt = oracle.bf16_round(np.sign(w) * np.float32(0.3)).astype(np.float64)
    xs = oracle.bf16_round(np.sign(x) * np.float32(0.8)).astype(np.float64)
    assert not np.allclose(g.astype(np.float64) @ wt, gx)                          # mask dropped
    assert not np.allclose((g.astype(np.float64) @ -wt) * o["middle"], gx)         # sign flipped
    wt_a = oracle.bf16_round(np.sign(w) * np.float32(0.8)).astype(np.float64)
    assert not np.allclose((g.astype(np.float64) @ wt_a) * o["middle"], gx)       # scales swapped
    mid_x = ((x >= -1) & (x <= 1)).astype(np.float64)
    assert not np.allclose((g.astype(np.float64) @ wt) * mid_x, gx)               # mask on x, not x / scale_a
    assert not np.allclose(g.astype(np.float64).T @ np.sign(x).astype(np.float64), gw)   # scale_a dropped
    assert not np.allclose(g.astype(np.float64).T @ oracle.bf16_round(np.sign(w[:M] if N >= M else w) * 0.8).astype(np.float64)[:, :K], gw)  # w for x


# ---------------------------------------------------------------------------
# Backward of the binary conv2d layer
# ---------------------------------------------------------------------------

def test_golden_conv_backward():
    for ex in json.load(open(GOLDEN))["conv_backward"]:
        o = oracle.conv2d_backward(np.array(ex["x"], np.float32), np.array(ex["w"], np.float32),
                                   np.array(ex["g"], np.float32), ex["scale_a"], ex["scale_w"], ex["stride"],
                                   ex["padding"], ex["dilation"], ex["x_dtype"])
        np.testing.assert_array_equal(o["grad_input"], np.array(ex["grad_input"], np.float32), ex["why"])
        np.testing.assert_array_equal(o["grad_weight"], np.array(ex["grad_weight"], np.float32), ex["why"])
        if "grad_scale_a" in ex:
            assert o["grad_scale_a"] == ex["grad_scale_a"], ex["why"]
        else:
            assert abs(o["grad_scale_a"] - 20.0 / 3.0) < 1e-6


def _conv_backward_scatter(x, w, g, scale_a, scale_w, s, p, d, mistake=None):
    """grad_input and grad_weight (exact, before rounding) by the definition
    of the convolution, summed output pixel by output pixel and tap by tap."""
    B, C, H, W = x.shape
    O, _, k, _ = w.shape
    _, _, Ho, Wo = g.shape
    wt = oracle.bf16_round(torch.from_numpy(w).sign().numpy() * np.float32(scale_w)).astype(np.float64)
    xs = oracle.bf16_round(torch.from_numpy(x).sign().numpy() * np.float32(scale_a)).astype(np.float64)
    gi = np.zeros((B, C, H, W))
    gw = np.zeros((O, C, k, k))
    for b, o, i, j in itertools.product(range(B), range(O), range(Ho), range(Wo)):
        gv = float(g[b, o, i, j])
        for c, kh, kw in itertools.product(range(C), range(k), range(k)):
            dd = 1 if mistake == "no_dilation" else d
            h, ww = i * s - p + kh * dd, j * s - p + kw * dd
            if 0 <= h < H and 0 <= ww < W:
                wv = wt[o, c, k - 1 - kh, k - 1 - kw] if mistake == "flipped_kernel" else wt[o, c, kh, kw]
                gi[b, c, h, ww] += gv * wv
                gw[o, c, kh, kw] += gv * xs[b, c, h, ww]
    return gi, gw


CONV_BWD_SHAPES = [(1, 2, 5, 5, 3, 3, 1, 1, 1), (2, 3, 6, 7, 2, 3, 2, 1, 1), (1, 2, 7, 6, 2, 3, 2, 2, 2),
                   (2, 1, 4, 4, 3, 1, 1, 0, 1), (1, 3, 5, 5, 2, 2, 3, 2, 1)]


@pytest.mark.parametrize("B,C,H,W,O,k,s,p,d", CONV_BWD_SHAPES)
def test_conv_backward_matches_scatter_loops(B, C, H, W, O, k, s, p, d):
    rng = np.random.default_rng(B * 1000 + C * 100 + H * 10 + k)
    ho, wo = oracle.conv2d_out_size(H, k, s, p, d), oracle.conv2d_out_size(W, k, s, p, d)
    x = torch.randn(B, C, H, W, generator=torch.Generator().manual_seed(H)).to(torch.bfloat16).float().numpy()
    w = rng.standard_normal((O, C, k, k)).astype(np.float32)
    g = torch.randn(B, O, ho, wo, generator=torch.Generator().manual_seed(W)).to(torch.bfloat16).float().numpy()
    o = oracle.conv2d_backward(x, w, g, 0.7, 0.4, s, p, d, "bf16")
    gi, gw = _conv_backward_scatter(x, w, g, 0.7, 0.4, s, p, d)
    np.testing.assert_allclose(o["grad_input_exact"], gi, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o["grad_weight_exact"], gw, rtol=0, atol=1e-12)


@pytest.mark.parametrize("B,C,H,W,O,k,s,p,d", CONV_BWD_SHAPES)
def test_conv_backward_matches_fold_unfold(B, C, H, W, O, k, s, p, d):
    # the unfold + mm lowering of banghao.live/blog/9 section 2, run backwards:
    # grad_input = fold(wt^T @ g), grad_weight = g @ unfold(xs)^T
    ho, wo = oracle.conv2d_out_size(H, k, s, p, d), oracle.conv2d_out_size(W, k, s, p, d)
    x = torch.randn(B, C, H, W, generator=torch.Generator().manual_seed(k)).to(torch.bfloat16).float().numpy()
    w = torch.randn(O, C, k, k, generator=torch.Generator().manual_seed(C)).numpy()
    g = torch.randn(B, O, ho, wo, generator=torch.Generator().manual_seed(O)).to(torch.bfloat16).float().numpy()
    o = oracle.conv2d_backward(x, w, g, 0.6, 0.3, s, p, d, "bf16")
    wt = torch.from_numpy(oracle.bf16_round(np.sign(w) * np.float32(0.3)).astype(np.float64)).reshape(O, -1)
    xs = torch.from_numpy(oracle.bf16_round(torch.from_numpy(x).sign().numpy() * np.float32(0.6)).astype(np.float64))
    gm = torch.from_numpy(g.astype(np.float64)).reshape(B, O, -1)
    cols = wt.T @ gm                                               # [B, C*k*k, L]
    gi = F.fold(cols, (H, W), k, dilation=d, padding=p, stride=s).numpy()
    u = F.unfold(xs, k, dilation=d, padding=p, stride=s)           # [B, C*k*k, L]
    gw = torch.einsum("bol,bcl->oc", gm, u).reshape(O, C, k, k).numpy()
    np.testing.assert_allclose(o["grad_input_exact"], gi, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o["grad_weight_exact"], gw, rtol=0, atol=1e-12)


def test_conv_backward_1x1_equals_linear_backward():
    B, C, O = 6, 9, 5
    x = torch.randn(B, C).to(torch.bfloat16).float().numpy()
    w = torch.randn(O, C).numpy().astype(np.float32)
    g = torch.randn(B, O).to(torch.bfloat16).float().numpy()
    oc = oracle.conv2d_backward(x[:, :, None, None], w[:, :, None, None], g[:, :, None, None], 0.8, 0.2, 1, 0, 1, "bf16")
    ol = oracle.linear_backward(x, w, g, 0.8, 0.2, "bf16")
    np.testing.assert_array_equal(oc["grad_input"][:, :, 0, 0], ol["grad_input"])
    np.testing.assert_array_equal(oc["grad_weight"][:, :, 0, 0], ol["grad_weight"])
    assert oc["grad_scale_a"] == ol["grad_scale_a"]


@pytest.mark.parametrize("mistake", ["flipped_kernel", "no_dilation"])
def test_planted_conv_backward_mistakes_are_caught(mistake):
    x = torch.randn(1, 2, 7, 7, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).float().numpy()
    w = torch.randn(2, 2, 3, 3, generator=torch.Generator().manual_seed(6)).numpy()
    g = torch.randn(1, 2, 3, 3, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16).float().numpy()
    o = oracle.conv2d_backward(x, w, g, 0.7, 0.4, 1, 0, 2, "bf16")
    gi, gw = _conv_backward_scatter(x, w, g, 0.7, 0.4, 1, 0, 2, mistake)
    assert not (np.allclose(o["grad_input_exact"], gi) and np.allclose(o["grad_weight_exact"], gw))


# ---------------------------------------------------------------------------
# Activation scale initialisation (set_activation)
# ---------------------------------------------------------------------------

def test_scale_init_hand_example():
    # |x| = [1, 3, 2, 2]: mean 2, symmetric factor 2 -> 4; asymmetric factor 4 -> 8
    x = np.array([1.0, -3.0, 2.0, -2.0], np.float32)
    assert oracle.scale_init(x, 2.0, "bf16", "bf16") == 4.0
    assert oracle.scale_init(x, 4.0, "f32", "f32") == 8.0
    # mean 1/3 in bf16: 0.333984375 (1.0101011b * 2^-2 rounded up), times 2 -> 0.66796875
    y = np.array([1.0, 0.0, 0.0], np.float32)
    assert oracle.scale_init(y, 2.0, "bf16", "bf16") == 0.66796875


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_scale_init_matches_torch_expression(dt):
    tdt = {"bf16": torch.bfloat16, "f32": torch.float32}[dt]
    for seed in range(5):
        x = torch.randn(1000 + 37 * seed, generator=torch.Generator().manual_seed(seed)).to(tdt)
        want = float((2 * x.abs().mean()).to(tdt))
        got = oracle.scale_init(x.float().numpy(), 2.0, dt, dt)
        step = abs(want) * (2.0 ** -7 if dt == "bf16" else 2.0 ** -23)
        assert abs(got - want) <= step          # torch accumulates in fp32; at most one rounding step apart


# ---------------------------------------------------------------------------
# W8A8 im2col + gemm convolution, with and without SmoothQuant
# ---------------------------------------------------------------------------

def test_golden_w8a8():
    for ex in json.load(open(GOLDEN))["w8a8_conv"]:
        o = oracle.w8a8_conv2d(np.array(ex["x"], np.float32), np.array(ex["w"], np.float32), ex["stride"],
                               ex["padding"], ex["dilation"], ex["smooth"])
        if "qx" in ex:
            np.testing.assert_array_equal(o["qx"], ex["qx"], ex["why"])
            np.testing.assert_array_equal(o["qw"], ex["qw"], ex["why"])
            np.testing.assert_array_equal(o["dot"], ex["dot"], ex["why"])
        if "balanced_max" in ex:
            np.testing.assert_allclose(np.abs(o["rows"]).max(0), ex["balanced_max"], rtol=3e-7)
            np.testing.assert_allclose(np.abs(o["wf"]).max(0), ex["balanced_max"], rtol=3e-7)


def test_fake_quant_matches_torch_fake_quantize():
    v = (torch.randn(5000, generator=torch.Generator().manual_seed(3)) * 3).numpy()
    v[:4] = [0.0, -0.0, 1e-6, -2.5]
    q, scale = oracle.fake_quant_int8(v)
    want = torch.fake_quantize_per_tensor_affine(torch.from_numpy(v), float(scale), 0, -127, 127).numpy()
    np.testing.assert_array_equal((q * np.float32(scale)).astype(np.float32), want)


@pytest.mark.parametrize("B,C,H,W,O,k,s,p,d", [(2, 3, 7, 6, 4, 3, 1, 1, 1), (1, 4, 9, 9, 3, 3, 2, 1, 1),
                                               (2, 2, 8, 8, 5, 3, 2, 2, 2), (1, 5, 5, 5, 2, 1, 1, 0, 1)])
def test_w8a8_integer_inputs_reduce_to_conv2d(B, C, H, W, O, k, s, p, d):
    # integer values with max |x| = max |w| = 127 quantize to themselves, so
    # the dot is the plain convolution of x and w
    rng = np.random.default_rng(B * 100 + C * 10 + k)
    x = rng.integers(-127, 128, (B, C, H, W)).astype(np.float32)
    w = rng.integers(-127, 128, (O, C, k, k)).astype(np.float32)
    x.flat[0], w.flat[0] = 127.0, -127.0
    o = oracle.w8a8_conv2d(x, w, s, p, d, smooth=False)
    ho, wo = oracle.conv2d_out_size(H, k, s, p, d), oracle.conv2d_out_size(W, k, s, p, d)
    want = F.conv2d(torch.from_numpy(x).double(), torch.from_numpy(w).double(), stride=s, padding=p,
                    dilation=d).numpy()
    dot = o["dot"].reshape(B, ho * wo, O).transpose(0, 2, 1).reshape(B, O, ho, wo)
    np.testing.assert_array_equal(dot, want)
    assert o["sx"] == np.float32(1.0) and o["sw"] == np.float32(1.0)
    np.testing.assert_array_equal(o["y"], want.astype(np.float32))


def test_w8a8_smooth_balances_column_maxima():
    x = (torch.randn(2, 6, 8, 8, generator=torch.Generator().manual_seed(8)) *
         torch.linspace(0.1, 20, 6).view(1, 6, 1, 1)).numpy()
    w = torch.randn(5, 6, 3, 3, generator=torch.Generator().manual_seed(9)).numpy()
    o = oracle.w8a8_conv2d(x, w, 1, 1, 1, smooth=True)
    np.testing.assert_allclose(np.abs(o["rows"]).max(0), np.abs(o["wf"]).max(0), rtol=5e-7)
    # migrating the scale leaves the unquantized product unchanged
    plain = oracle.w8a8_conv2d(x, w, 1, 1, 1, smooth=False)
    np.testing.assert_allclose(o["rows"].astype(np.float64) @ o["wf"].T.astype(np.float64),
                               plain["rows"].astype(np.float64) @ plain["wf"].T.astype(np.float64), rtol=1e-5,
                               atol=1e-4)


@pytest.mark.parametrize("smooth", [False, True])
def test_w8a8_at_agrees_with_full(smooth):
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((2, 5, 9, 8)) * np.logspace(-1, 1, 5)[None, :, None, None]).astype(np.float32)
    w = rng.standard_normal((6, 5, 3, 3)).astype(np.float32)
    full = oracle.w8a8_conv2d(x, w, 2, 1, 1, smooth)["y"]
    flat = np.arange(full.size)
    np.testing.assert_array_equal(oracle.w8a8_conv2d_at(x, w, 2, 1, 1, smooth, flat), full.reshape(-1))


@pytest.mark.parametrize("s,p,d", [(1, 1, 1), (2, 1, 1), (2, 2, 2)])
def test_conv2d_grad_weight_at_agrees_with_full(s, p, d):
    rng = np.random.default_rng(13)
    x = rng.standard_normal((2, 3, 9, 8)).astype(np.float32)
    w = rng.standard_normal((4, 3, 3, 3)).astype(np.float32)
    ho, wo = oracle.conv2d_out_size(9, 3, s, p, d), oracle.conv2d_out_size(8, 3, s, p, d)
    g = oracle.bf16_round(rng.standard_normal((2, 4, ho, wo)).astype(np.float32))
    full = oracle.conv2d_backward(x, w, g, 0.7, 0.3, s, p, d, "f32")["grad_weight_exact"].reshape(4, -1)
    o_idx, t_idx = np.meshgrid(np.arange(4), np.arange(27), indexing="ij")
    got = oracle.conv2d_grad_weight_at(x, g, 0.7, s, p, d, 3, o_idx.ravel(), t_idx.ravel())
    np.testing.assert_array_equal(got, full.ravel())
