"""GPU: the implicit-im2col tensor-core convolution against the CPU oracle.

The convolution reads channel-packed NHWC pixels in place: each filter tap is
a shifted view of one staged image per stride phase, so no im2col matrix is
written. Integer outputs must equal oracle.conv2d_dot bit for bit and scaled
outputs oracle.binary_conv2d within 1e-6 relative. The geometries cover both
slice widths (64- and 128-byte rows of codes), taps of several slices,
strides 1 and 2 with every padding/dilation phase pattern, one and many
bands of output rows per image, channel counts that are not a multiple of the
128-channel tile, weights kept resident and weights streamed per tile, and
inputs smaller than one staged image. The explicit unfold
(BT_CONV_IMPLICIT=0) stays under test beside it. Float inputs take the route
through the NHWC pack kernel here (BT_CONV_FUSED=0); the convolution that
packs x itself has its own tests.
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
XT = {torch.float32: bt.BT_F32, torch.bfloat16: bt.BT_BF16}


@pytest.fixture(autouse=True)
def _device_clean():
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


def _implicit(B, C, H, W, k, s, p, d, code):
    """True when the library contracts the packed pixels in place for this
    geometry: it then needs no workspace for packed input."""
    return bt.bt_binary_conv2d_workspace(B, C, H, W, k, s, p, d, bt.BT_PACKED, code) == 0


SHAPES = [
    # B, C, H, W, O, k, s, p, d
    (2, 128, 14, 14, 256, 3, 1, 1, 1),     # 64-byte E2M1 slices, one band
    (2, 256, 14, 14, 200, 3, 1, 1, 1),     # 128-byte E2M1 slices, weights streamed
    (3, 128, 28, 28, 130, 3, 2, 1, 1),     # stride 2: four phase images
    (3, 128, 28, 28, 64, 3, 2, 2, 2),      # stride 2, dilation 2: one phase image
    (2, 64, 30, 33, 70, 3, 1, 1, 1),       # several bands per image
    (1, 96, 57, 23, 40, 5, 2, 2, 1),       # 5x5, odd sizes, bands
    (2, 384, 9, 9, 33, 3, 1, 1, 1),        # three 64-byte slices per tap
    (2, 512, 7, 7, 129, 3, 1, 1, 1),       # two 128-byte slices per tap
    (1, 3, 5, 5, 4, 3, 1, 1, 1),           # tiny C
    (2, 40, 1, 1, 17, 3, 1, 1, 1),         # 1x1 image: only the centre tap inside
    (2, 33, 8, 8, 7, 1, 1, 0, 1),          # 1x1 kernel
    (1, 70, 13, 13, 130, 3, 2, 1, 2),      # stride 2, dilation 2, padding 1: two phases
    (1, 40, 12, 10, 33, 3, 2, 0, 1),       # stride 2, no padding
    (2, 64, 11, 11, 48, 7, 1, 3, 1),       # 7x7
    (1, 32, 20, 200, 16, 3, 1, 1, 1),      # wide rows: one output row per band
]


@pytest.mark.parametrize("pair", ["1", "0"], ids=["pair", "single"])
@pytest.mark.parametrize("code", TC_CODES, ids=TC_IDS)
@pytest.mark.parametrize("B,C,H,W,O,k,s,p,d", SHAPES)
def test_implicit_conv_matches_oracle(code, B, C, H, W, O, k, s, p, d, pair, monkeypatch):
    # pair: clusters of two CTAs, 256-channel tiles, half of a band's rows per
    # CTA (where that plan fits); single: one CTA per 128-channel tile
    monkeypatch.setenv("BT_CONV_FUSED", "0")
    monkeypatch.setenv("BT_CONV_PAIR", pair)
    assert _implicit(B, C, H, W, k, s, p, d, code)
    x = _gen(B * 7 + C + H, (B, C, H, W), torch.bfloat16)
    w = _gen(O + k + C, (O, C, k, k), torch.bfloat16)
    bias = torch.linspace(-0.1, 0.1, C)
    sa, sw = workloads.mean_abs(x), workloads.mean_abs(w)
    sx = oracle.binarize(x, bias, channel_axis=1)
    want = oracle.conv2d_dot(sx, oracle.binarize_weight(w), s, p, d)
    wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    xd = x.to(DEV)
    for od in ("i32", "f32", "bf16"):
        got = bt.bt_binary_conv2d(xd, wp, code, C, k, s, p, d, sa, sw, bias.to(DEV), out_dtype=OUT_T[od]).cpu()
        _close(got, oracle.epilogue(want, sa, sw, od))
    # packed pixels in, no workspace
    xp = bt.bt_pack_sign(xd, code, bt.BT_LAYOUT_NCHW_TO_NHWC, bias.to(DEV))
    got = bt.bt_binary_conv2d(xp, wp, code, C, k, s, p, d, 1.0, 1.0, out_dtype=torch.int32, x_packed=True).cpu()
    assert torch.equal(got, torch.from_numpy(want))


@pytest.mark.parametrize("code", TC_CODES, ids=TC_IDS)
@pytest.mark.parametrize("B,C,H,W,O,k,s,p,d", [SHAPES[0], SHAPES[2], SHAPES[3], SHAPES[4]])
def test_explicit_unfold_still_matches_oracle(code, B, C, H, W, O, k, s, p, d, monkeypatch):
    monkeypatch.setenv("BT_CONV_IMPLICIT", "0")
    assert not _implicit(B, C, H, W, k, s, p, d, code)
    x = _gen(B + C, (B, C, H, W), torch.bfloat16)
    w = _gen(O + C, (O, C, k, k), torch.bfloat16)
    want = oracle.conv2d_dot(oracle.binarize(x), oracle.binarize_weight(w), s, p, d)
    wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    got = bt.bt_binary_conv2d(x.to(DEV), wp, code, C, k, s, p, d, 1.0, 1.0, out_dtype=torch.int32).cpu()
    assert torch.equal(got, torch.from_numpy(want))


@pytest.mark.parametrize("code", TC_CODES, ids=TC_IDS)
def test_implicit_conv_extreme_sums(code):
    # all-equal signs drive every interior dot to +-C*k*k and border dots to
    # +-C * (taps inside): exact at the largest magnitudes the tiles produce
    B, C, H, W, O, k = 2, 256, 9, 9, 130, 3
    x = torch.ones(B, C, H, W)
    x[1] = -1.0
    w = torch.ones(O, C, k, k)
    w[::2] = -1.0
    want = oracle.conv2d_dot(oracle.binarize(x), oracle.binarize_weight(w), 1, 1, 1)
    wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    got = bt.bt_binary_conv2d(x.to(DEV), wp, code, C, k, 1, 1, 1, 1.0, 1.0, out_dtype=torch.int32).cpu()
    assert torch.equal(got, torch.from_numpy(want))
    assert int(got.abs().max()) == C * k * k


def test_single_pass_query_follows_the_implicit_path(monkeypatch):
    # where the contraction reads packed pixels in place, the library's own
    # split is pack (NHWC) + contraction (or, opted in, one kernel from x with
    # 16-byte channel planes), never the one-pass unfold
    for (B, C, H, W, k, s, p, d) in ((256, 128, 28, 28, 3, 2, 1, 1), (128, 256, 14, 14, 3, 1, 1, 1)):
        for code in TC_CODES:
            assert _implicit(B, C, H, W, k, s, p, d, code)
            assert bt.bt_conv2d_single_pass(B, C, H, W, k, s, p, d, bt.BT_BF16, code) == 0
            fused = (H * W * 2) % 16 == 0
            monkeypatch.setenv("BT_CONV_FUSED", "1")
            assert bt.bt_conv2d_single_pass(B, C, H, W, k, s, p, d, bt.BT_BF16, code) == (2 if fused else 0)
            monkeypatch.delenv("BT_CONV_FUSED")


@pytest.mark.parametrize("code", TC_CODES, ids=TC_IDS)
def test_rows_too_wide_for_one_tile_take_the_explicit_unfold(code):
    B, C, H, W, O, k, s, p, d = 1, 16, 3, 300, 8, 3, 1, 1, 1
    assert not _implicit(B, C, H, W, k, s, p, d, code)
    x = _gen(3, (B, C, H, W), torch.bfloat16)
    w = _gen(4, (O, C, k, k), torch.bfloat16)
    want = oracle.conv2d_dot(oracle.binarize(x), oracle.binarize_weight(w), s, p, d)
    wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    got = bt.bt_binary_conv2d(x.to(DEV), wp, code, C, k, s, p, d, 1.0, 1.0, out_dtype=torch.int32).cpu()
    assert torch.equal(got, torch.from_numpy(want))


@pytest.mark.parametrize("code", TC_CODES, ids=TC_IDS)
def test_weights_packed_just_before_each_call(code):
    # After the library's own pack of x, the convolution may start its weight
    # copies before it waits on that pack; the pack of x lets it start only once
    # its own wait is over, so weights written by the kernel before (here a
    # weight pack into the same buffer, right before every call) are complete
    # by then. Every call must see the weights packed for it.
    B, C, H, W, O, k, s, p, d = 4, 128, 28, 28, 256, 3, 2, 1, 1
    x = _gen(51, (B, C, H, W), torch.bfloat16)
    ws = [_gen(52 + i, (O, C, k, k), torch.bfloat16) for i in range(3)]
    xd = x.to(DEV)
    wbuf = bt.bt_pack_sign(ws[0].to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    wds = [w.to(DEV) for w in ws]
    torch.cuda.synchronize()
    outs = []
    for i in range(6):
        bt.bt_pack_sign(wds[i % 3], code, bt.BT_LAYOUT_NCHW_TO_NHWC, out=wbuf)
        outs.append(bt.bt_binary_conv2d(xd, wbuf, code, C, k, s, p, d, 1.0, 1.0, out_dtype=torch.int32))
    torch.cuda.synchronize()
    sx = oracle.binarize(x)
    wants = [oracle.conv2d_dot(sx, oracle.binarize_weight(w), s, p, d) for w in ws]
    for i, got in enumerate(outs):
        assert torch.equal(got.cpu(), torch.from_numpy(wants[i % 3]))


@pytest.mark.parametrize("split", ["2", "4"])
@pytest.mark.parametrize("pair", ["1", "0"], ids=["pair", "single"])
@pytest.mark.parametrize("code", TC_CODES, ids=TC_IDS)
@pytest.mark.parametrize("B,C,H,W,O,k,s,p,d", [SHAPES[0], SHAPES[2], SHAPES[3], SHAPES[4], SHAPES[5], SHAPES[13]])
def test_implicit_conv_more_bands_matches_oracle(code, B, C, H, W, O, k, s, p, d, pair, split, monkeypatch):
    # BT_CONV_SPLIT: each image cut into 2 or 4 times the bands that fit a
    # tile (narrower tiles, as the measured selection may keep), packed pixels
    # read in place
    monkeypatch.setenv("BT_CONV_FUSED", "0")
    monkeypatch.setenv("BT_CONV_PAIR", pair)
    monkeypatch.setenv("BT_CONV_SPLIT", split)
    assert _implicit(B, C, H, W, k, s, p, d, code)
    x = _gen(B * 5 + C + H, (B, C, H, W), torch.bfloat16)
    w = _gen(O + k + 3 * C, (O, C, k, k), torch.bfloat16)
    want = oracle.conv2d_dot(oracle.binarize(x), oracle.binarize_weight(w), s, p, d)
    wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    sa, sw = workloads.mean_abs(x), workloads.mean_abs(w)
    for od in ("i32", "bf16"):
        got = bt.bt_binary_conv2d(x.to(DEV), wp, code, C, k, s, p, d, sa, sw, out_dtype=OUT_T[od]).cpu()
        _close(got, oracle.epilogue(want, sa, sw, od))


@pytest.mark.parametrize("split", ["2", "4"])
@pytest.mark.parametrize("pair", ["1", "0"], ids=["pair", "single"])
@pytest.mark.parametrize("fused", ["0", "1"], ids=["packed", "fused"])
@pytest.mark.parametrize("code", TC_CODES, ids=TC_IDS)
def test_more_bands_several_tiles_per_cta(code, fused, pair, split, monkeypatch):
    # enough images that CTAs take three or more tiles each, so both
    # accumulator buffers are reused after bands whose last rows leave some
    # epilogue warps without a box (the 14-row image cut into 4 bands of 4,
    # 4, 4 and 2 rows): every warp must still hand the buffer back
    monkeypatch.setenv("BT_CONV_FUSED", fused)
    monkeypatch.setenv("BT_CONV_PAIR", pair)
    monkeypatch.setenv("BT_CONV_SPLIT", split)
    # (f32 x: 784-byte channel planes, so the convolution that packs x itself applies)
    B, C, H, W, O, k, s, p, d = 48, 128, 14, 14, 256, 3, 1, 1, 1
    x = _gen(B + 77, (B, C, H, W), torch.float32)
    w = _gen(O + 78, (O, C, k, k), torch.float32)
    want = oracle.conv2d_dot(oracle.binarize(x), oracle.binarize_weight(w), s, p, d)
    wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    got = bt.bt_binary_conv2d(x.to(DEV), wp, code, C, k, s, p, d, 1.0, 1.0, out_dtype=torch.int32).cpu()
    assert bt.bt_device_status() == 0
    assert torch.equal(got, torch.from_numpy(want))


@pytest.mark.parametrize("pair", ["1", "0"], ids=["pair", "single"])
@pytest.mark.parametrize("code", TC_CODES, ids=TC_IDS)
@pytest.mark.parametrize("B,C,H,W,O", [(400, 40, 1, 1, 17), (360, 64, 3, 3, 96)])
def test_tiny_images_several_tiles_per_cta(code, B, C, H, W, O, pair, monkeypatch):
    # images whose whole band fits one 32-column epilogue box, many of them:
    # CTAs take three tiles or more, and the epilogue warps without a box must
    # still hand each accumulator buffer back
    monkeypatch.setenv("BT_CONV_FUSED", "0")
    monkeypatch.setenv("BT_CONV_PAIR", pair)
    k, s, p, d = 3, 1, 1, 1
    assert _implicit(B, C, H, W, k, s, p, d, code)
    x = _gen(B + H, (B, C, H, W), torch.bfloat16)
    w = _gen(O + C, (O, C, k, k), torch.bfloat16)
    want = oracle.conv2d_dot(oracle.binarize(x), oracle.binarize_weight(w), s, p, d)
    wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    got = bt.bt_binary_conv2d(x.to(DEV), wp, code, C, k, s, p, d, 1.0, 1.0, out_dtype=torch.int32).cpu()
    assert bt.bt_device_status() == 0
    assert torch.equal(got, torch.from_numpy(want))
