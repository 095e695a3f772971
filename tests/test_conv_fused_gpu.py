"""GPU: the tensor-core convolution that packs its own input, against the CPU oracle.

With BT_CONV_FUSED=1, where the implicit-im2col plan applies and every channel
plane of x is a whole number of 16-byte units, bt_binary_conv2d on float x is
one kernel: its packing
warps read x, shift it by bias_a, take the sign and write the channel-packed
codes straight into the shared-memory pixel stages the tensor core reads. The
shift + sign is that of bitorch-engine BinaryConv2dCutlass.set_activation (x +
bias_a.view(1, -1, 1, 1) >= 0 is +1), the contraction and epilogue those of
BinaryConv2dForward.forward. Integer outputs must equal oracle.conv2d_dot bit
for bit, scaled ones oracle.binary_conv2d within 1e-6 relative.

Both tile shapes run: CTA pairs (256 output channels per tile, each CTA
packing and staging half the rows of a band) and single CTAs. The geometries
cover strides 1 and 2 (one to four phase images, and parities
that no tap reads), several bands of output rows per image (staged rows past
the image cleared per tile), channel counts that are not a multiple of 32,
64- and 128-byte slices, several slices per tap, weights resident and
streamed, one and two pixel stages; the inputs f32, bf16 and f16 with no
shift, one shift, a shift per channel, and infinite shifts.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import xnor_popcount_gemm_gb300 as bt

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
REL_TOL = 1e-6
OUT_T = {"f32": torch.float32, "bf16": torch.bfloat16, "i32": torch.int32}
TC_CODES = [bt.BT_CODE_E4M3, bt.BT_CODE_E2M1]
TC_IDS = ["e4m3", "e2m1"]
XT = {torch.float32: bt.BT_F32, torch.bfloat16: bt.BT_BF16, torch.float16: bt.BT_F16}


@pytest.fixture(autouse=True)
def _device_clean(monkeypatch):
    # the fused route is opt-in (BT_CONV_FUSED=1); every test here runs it
    monkeypatch.setenv("BT_CONV_FUSED", "1")
    yield
    assert bt.bt_device_status() == 0


def _gen(seed, shape, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(dtype)


def _close(got, want):
    assert got.shape == want.shape and got.dtype == want.dtype
    if got.dtype == torch.int32:
        assert torch.equal(got, want)
        return
    err = (got.double() - want.double()).abs()
    assert not (err > REL_TOL * want.double().abs()).any()


def _mode(x, C, k, s, p, d, code):
    B, _, H, W = x.shape
    return bt.bt_conv2d_single_pass(B, C, H, W, k, s, p, d, XT[x.dtype], code)


SHAPES = [
    # B, C, H, W, O, k, s, p, d
    (2, 128, 16, 16, 256, 3, 1, 1, 1),     # 64-byte E2M1 slices, one band
    (2, 256, 14, 14, 200, 3, 1, 1, 1),     # 128-byte slices (f32 planes only: 784 bytes)
    (3, 128, 28, 28, 130, 3, 2, 1, 1),     # stride 2: four phase images
    (3, 128, 28, 28, 64, 3, 2, 2, 2),      # stride 2, dilation 2: one phase image, odd rows unread
    (2, 64, 32, 32, 70, 3, 1, 1, 1),       # five bands per image
    (1, 96, 56, 24, 40, 5, 2, 2, 1),       # 5x5, stride 2, two bands
    (2, 384, 8, 8, 33, 3, 1, 1, 1),        # three 64-byte slices per tap
    (2, 512, 8, 8, 129, 3, 1, 1, 1),       # two 128-byte slices per tap
    (1, 3, 8, 8, 4, 3, 1, 1, 1),           # three channels
    (2, 40, 8, 8, 17, 3, 1, 1, 1),         # a partial 32-channel group
    (2, 33, 8, 8, 7, 1, 1, 0, 1),          # 1x1 kernel
    (2, 64, 16, 16, 48, 1, 2, 0, 1),       # 1x1 stride 2: three parities unread
    (1, 70, 16, 16, 130, 3, 2, 1, 2),      # stride 2, dilation 2, padding 1: two phases
    (1, 40, 12, 12, 33, 3, 2, 0, 1),       # stride 2, no padding
    (2, 64, 12, 12, 48, 7, 1, 3, 1),       # 7x7
    (1, 32, 20, 200, 16, 3, 1, 1, 1),      # wide rows: one output row per band
    (5, 64, 8, 8, 300, 3, 1, 1, 1),        # three channel tiles
]


@pytest.mark.parametrize("pair", ["1", "0"], ids=["pair", "single"])
@pytest.mark.parametrize("code", TC_CODES, ids=TC_IDS)
@pytest.mark.parametrize("B,C,H,W,O,k,s,p,d", SHAPES)
def test_fused_conv_matches_oracle(code, B, C, H, W, O, k, s, p, d, pair, monkeypatch):
    # pair: clusters of two CTAs with 256-channel tiles (each CTA half the
    # rows of a band) wherever that plan fits; single: one CTA per tile
    monkeypatch.setenv("BT_CONV_PAIR", pair)
    w = _gen(O + k + C, (O, C, k, k), torch.bfloat16)
    wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    sw_ = oracle.binarize_weight(w)
    ran = 0
    for dt in (torch.float32, torch.bfloat16, torch.float16):
        x = _gen(B * 7 + C + H + dt.itemsize, (B, C, H, W), dt)
        if _mode(x, C, k, s, p, d, code) != 2:
            assert (H * W * dt.itemsize) % 16 != 0     # only misaligned planes leave the fused route
            continue
        ran += 1
        bias = torch.linspace(-0.1, 0.1, C)
        sa, sw = workloads.mean_abs(x), workloads.mean_abs(w)
        want = oracle.conv2d_dot(oracle.binarize(x, bias, channel_axis=1), sw_, s, p, d)
        xd = x.to(DEV)
        for od in ("i32", "f32", "bf16"):
            got = bt.bt_binary_conv2d(xd, wp, code, C, k, s, p, d, sa, sw, bias.to(DEV), out_dtype=OUT_T[od]).cpu()
            _close(got, oracle.epilogue(want, sa, sw, od))
        # one shift for every channel, and none
        for b1 in (torch.tensor([0.05]), None):
            want = oracle.conv2d_dot(oracle.binarize(x, b1), sw_, s, p, d)
            got = bt.bt_binary_conv2d(xd, wp, code, C, k, s, p, d, 1.0, 1.0, None if b1 is None else b1.to(DEV),
                                      out_dtype=torch.int32).cpu()
            assert torch.equal(got, torch.from_numpy(want))
    assert ran > 0


@pytest.mark.parametrize("code", TC_CODES, ids=TC_IDS)
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16, torch.float16], ids=["f32", "bf16", "f16"])
def test_fused_conv_shift_edges(code, dt):
    # values exactly at -bias (binarize to +1), signed zeros, infinities, and
    # infinite shifts (every value of the channel +1 or -1)
    B, C, H, W, O, k, s, p, d = 2, 64, 16, 16, 40, 3, 2, 1, 1
    x = _gen(11, (B, C, H, W)).to(dt)
    bias = torch.linspace(-0.5, 0.5, C).to(dt).float()     # representable in dt: x == -bias is reachable
    x[:, :, 0, :] = (-bias).to(dt).view(1, C, 1)
    x[:, :, 1, :] = -0.0
    x[:, :, 2, 0] = float("inf")
    x[:, :, 2, 1] = float("-inf")
    bias[3] = float("inf")
    bias[4] = float("-inf")
    w = _gen(12, (O, C, k, k))
    wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    assert _mode(x, C, k, s, p, d, code) == 2
    want = oracle.conv2d_dot(oracle.binarize(x, bias, channel_axis=1), oracle.binarize_weight(w), s, p, d)
    got = bt.bt_binary_conv2d(x.to(DEV), wp, code, C, k, s, p, d, 1.0, 1.0, bias.to(DEV), out_dtype=torch.int32)
    assert torch.equal(got.cpu(), torch.from_numpy(want))


@pytest.mark.parametrize("pair", ["1", "0"], ids=["pair", "single"])
@pytest.mark.parametrize("code", TC_CODES, ids=TC_IDS)
@pytest.mark.parametrize("plan", ["r2", "r1", "s2", "s1"])
def test_fused_conv_every_plan(code, plan, pair, monkeypatch):
    # weights resident or streamed, two pixel stages or one: the packing warps
    # and the MMA issuer hand the stages back and forth the same way
    monkeypatch.setenv("BT_CONV_PLAN", plan)
    monkeypatch.setenv("BT_CONV_PAIR", pair)
    B, C, H, W, O, k, s, p, d = 7, 128, 16, 16, 256, 3, 1, 1, 1
    x = _gen(21, (B, C, H, W), torch.bfloat16)
    w = _gen(22, (O, C, k, k))
    assert _mode(x, C, k, s, p, d, code) == 2
    wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    want = oracle.conv2d_dot(oracle.binarize(x), oracle.binarize_weight(w), s, p, d)
    got = bt.bt_binary_conv2d(x.to(DEV), wp, code, C, k, s, p, d, 1.0, 1.0, out_dtype=torch.int32)
    assert torch.equal(got.cpu(), torch.from_numpy(want))


@pytest.mark.parametrize("code", TC_CODES, ids=TC_IDS)
def test_fused_and_two_kernel_routes_agree_with_the_oracle(code, monkeypatch):
    # the same call with the fused route turned off (NHWC pack, then the
    # implicit contraction of packed pixels): both equal the oracle
    B, C, H, W, O, k, s, p, d = 4, 128, 28, 28, 256, 3, 2, 1, 1
    x = _gen(31, (B, C, H, W), torch.bfloat16)
    w = _gen(32, (O, C, k, k))
    bias = torch.linspace(-0.2, 0.2, C)
    wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    want = oracle.conv2d_dot(oracle.binarize(x, bias, channel_axis=1), oracle.binarize_weight(w), s, p, d)
    for fused in ("1", "0"):
        monkeypatch.setenv("BT_CONV_FUSED", fused)
        assert _mode(x, C, k, s, p, d, code) == (2 if fused == "1" else 0)
        got = bt.bt_binary_conv2d(x.to(DEV), wp, code, C, k, s, p, d, 1.0, 1.0, bias.to(DEV), out_dtype=torch.int32)
        assert torch.equal(got.cpu(), torch.from_numpy(want))


def test_fused_conv_needs_no_workspace():
    B, C, H, W, O, k = 2, 128, 16, 16, 64, 3
    x = _gen(41, (B, C, H, W), torch.bfloat16).to(DEV)
    w = _gen(42, (O, C, k, k))
    code = bt.BT_CODE_E2M1
    wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    out = torch.empty(B, O, H, W, dtype=torch.int32, device=DEV)
    st = bt._c_conv(bt._ptr(x), bt.BT_BF16, bt._ptr(wp), code, B, C, H, W, O, k, 1, 1, 1, 1.0, 1.0, None, 0,
                    bt._ptr(out), bt.BT_I32, bt.BT_ALGO_AUTO, None, 0, None)
    assert st == bt.BT_OK
    want = oracle.conv2d_dot(oracle.binarize(x.cpu()), oracle.binarize_weight(w), 1, 1, 1)
    assert torch.equal(out.cpu(), torch.from_numpy(want))


@pytest.mark.parametrize("split", ["2", "4"])
@pytest.mark.parametrize("pair", ["1", "0"], ids=["pair", "single"])
@pytest.mark.parametrize("code", TC_CODES, ids=TC_IDS)
def test_fused_conv_more_bands(code, pair, split, monkeypatch):
    # the convolution that packs x itself over 2 or 4 times the bands: staged
    # rows past the image are cleared per tile
    monkeypatch.setenv("BT_CONV_FUSED", "1")
    monkeypatch.setenv("BT_CONV_PAIR", pair)
    monkeypatch.setenv("BT_CONV_SPLIT", split)
    for (B, C, H, W, O, k, s, p, d) in ((3, 128, 16, 16, 256, 3, 1, 1, 1), (2, 128, 28, 28, 130, 3, 2, 1, 1)):
        x = _gen(41 + H, (B, C, H, W), torch.bfloat16)
        w = _gen(42 + O, (O, C, k, k))
        bias = torch.linspace(-0.2, 0.2, C)
        assert _mode(x, C, k, s, p, d, code) == 2
        wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
        want = oracle.conv2d_dot(oracle.binarize(x, bias, channel_axis=1), oracle.binarize_weight(w), s, p, d)
        got = bt.bt_binary_conv2d(x.to(DEV), wp, code, C, k, s, p, d, 1.0, 1.0, bias.to(DEV), out_dtype=torch.int32)
        assert torch.equal(got.cpu(), torch.from_numpy(want))
