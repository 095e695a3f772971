"""GPU parity of the W8A8 im2col + gemm convolution (with and without
SmoothQuant) against oracle.w8a8_conv2d. Both sides take the same fp32 steps
(column maxima, sqrt scales, per-tensor maxima, fp32(1 / scale), round half
to even, clamp), the integer dot products are exact on both, and the output
is one double product rounded to fp32: the outputs must be bit-identical."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import xnor_popcount_gemm_gb300 as bt

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _device_clean():
    yield
    assert bt.bt_device_status() == 0


SHAPES = [(2, 8, 9, 9, 16, 3, 1, 1, 1), (3, 5, 11, 10, 24, 3, 2, 1, 1), (2, 16, 12, 12, 32, 3, 2, 2, 2),
          (1, 3, 7, 7, 8, 1, 1, 0, 1), (2, 130, 14, 14, 40, 3, 1, 1, 1), (1, 4, 6, 6, 12, 5, 1, 2, 1),
          (2, 20, 15, 13, 17, 3, 3, 1, 1)]


@pytest.mark.parametrize("B,C,H,W,O,k,s,p,d", SHAPES)
@pytest.mark.parametrize("smooth", [False, True], ids=["plain", "smoothquant"])
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_w8a8_matches_oracle(B, C, H, W, O, k, s, p, d, smooth, dt):
    gen = torch.Generator().manual_seed(B * 1000 + C + k)
    # channels of very different ranges, the case SmoothQuant is for
    x = (torch.randn(B, C, H, W, generator=gen) * torch.logspace(-1, 1.5, C).view(1, C, 1, 1)).to(dt)
    w = (torch.randn(O, C, k, k, generator=gen) * 0.1).to(dt)
    got = bt.bt_w8a8_conv2d(x.to(DEV), w.to(DEV), s, p, d, smooth=smooth).cpu().numpy()
    want = oracle.w8a8_conv2d(x.float().numpy(), w.float().numpy(), s, p, d, smooth)["y"]
    assert got.shape == want.shape
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("B,C,H,W,O,k,s,p,d", SHAPES[:4] + [(1, 7, 40, 40, 8, 3, 1, 0, 12)])
@pytest.mark.parametrize("smooth", [False, True], ids=["plain", "smoothquant"])
def test_w8a8_direct_gather_matches_oracle(B, C, H, W, O, k, s, p, d, smooth, monkeypatch):
    # the direct gather (forced here; the last shape's dilated window fits no
    # staged plan, so it takes the gather on its own) gives the same rows
    monkeypatch.setenv("BT_W8A8_UNFOLD", "gather")
    gen = torch.Generator().manual_seed(B * 1000 + C + k + 1)
    x = (torch.randn(B, C, H, W, generator=gen) * torch.logspace(-1, 1.5, C).view(1, C, 1, 1)).to(torch.bfloat16)
    w = (torch.randn(O, C, k, k, generator=gen) * 0.1).to(torch.bfloat16)
    got = bt.bt_w8a8_conv2d(x.to(DEV), w.to(DEV), s, p, d, smooth=smooth).cpu().numpy()
    want = oracle.w8a8_conv2d(x.float().numpy(), w.float().numpy(), s, p, d, smooth)["y"]
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("B,C,H,W,O,k,s,p,d", [(1, 7, 40, 40, 8, 3, 1, 0, 12), (1, 3, 33, 33, 8, 8, 1, 3, 1),
                                               (1, 5, 30, 30, 8, 7, 1, 3, 1), (1, 33, 5, 150, 8, 3, 2, 1, 1),
                                               (1, 300, 4, 4, 8, 1, 1, 0, 1), (2, 40, 9, 9, 8, 2, 1, 0, 1)])
def test_w8a8_unusual_windows_match_oracle(B, C, H, W, O, k, s, p, d):
    # dilated windows too wide to stage, 7x7 and 8x8 kernels (fewer pixel
    # slots per unit), wide rows split in column ranges, 1x1 and 2x2 kernels
    # (more channels per unit)
    gen = torch.Generator().manual_seed(C * 7 + k)
    x = torch.randn(B, C, H, W, generator=gen)
    w = torch.randn(O, C, k, k, generator=gen)
    got = bt.bt_w8a8_conv2d(x.to(DEV), w.to(DEV), s, p, d, smooth=True).cpu().numpy()
    want = oracle.w8a8_conv2d(x.numpy(), w.numpy(), s, p, d, True)["y"]
    np.testing.assert_array_equal(got, want)


def test_w8a8_bf16_output_and_large_k():
    # C*k*k = 2304 taps: three K splits, each exact in fp32
    gen = torch.Generator().manual_seed(5)
    x = torch.randn(2, 256, 14, 14, generator=gen).to(torch.bfloat16)
    w = (torch.randn(64, 256, 3, 3, generator=gen) * 0.05).to(torch.bfloat16)
    got = bt.bt_w8a8_conv2d(x.to(DEV), w.to(DEV), 1, 1, 1, smooth=True, out_dtype=torch.bfloat16).cpu()
    want = oracle.w8a8_conv2d(x.float().numpy(), w.float().numpy(), 1, 1, 1, True)["y"]
    assert torch.equal(got, torch.from_numpy(want).to(torch.bfloat16))


def test_w8a8_extreme_integer_sums_are_exact():
    # every product +127 * 127 over K = 2304 taps: |dot| = 2304 * 16129 > 2^24,
    # exact only because each K split stays below 2^24
    x = torch.full((1, 256, 5, 5), 3.0)
    w = torch.full((8, 256, 3, 3), -2.0)
    got = bt.bt_w8a8_conv2d(x.to(DEV), w.to(DEV), 1, 0, 1).cpu().numpy()
    o = oracle.w8a8_conv2d(x.numpy(), w.numpy(), 1, 0, 1, False)
    assert int(np.abs(o["dot"]).max()) == 2304 * 127 * 127
    np.testing.assert_array_equal(got, o["y"])


@pytest.mark.parametrize("unfold", ["staged", "gather"])
def test_w8a8_rounding_ties_to_even(unfold, monkeypatch):
    # max|x| = 127, so the input scale is 1 and x * (1 / scale) = x: every
    # other value is an exact tie k + 1/2, which rounds to even on both sides
    if unfold == "gather":
        monkeypatch.setenv("BT_W8A8_UNFOLD", "gather")
    ties = torch.tensor([0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, 126.5, -126.5, 63.5, -64.5, 127.0])
    x = ties.repeat(2 * 3 * 6 * 6 // ties.numel()).view(2, 3, 6, 6)
    gen = torch.Generator().manual_seed(11)
    w = torch.randn(8, 3, 3, 3, generator=gen)
    got = bt.bt_w8a8_conv2d(x.to(DEV), w.to(DEV), 1, 1, 1).cpu().numpy()
    o = oracle.w8a8_conv2d(x.numpy(), w.numpy(), 1, 1, 1, False)
    assert float(o["sx"]) == 1.0
    np.testing.assert_array_equal(got, o["y"])


def test_w8a8_zero_input_and_empty_batch():
    x = torch.zeros(2, 8, 6, 6, device=DEV)
    w = torch.randn(16, 8, 3, 3, device=DEV)
    assert torch.all(bt.bt_w8a8_conv2d(x, w, 1, 1, 1).cpu() == 0)
    e = bt.bt_w8a8_conv2d(torch.empty(0, 8, 6, 6, device=DEV), w, 1, 1, 1)
    assert e.shape == (0, 16, 6, 6)


@pytest.mark.slow
@pytest.mark.parametrize("smooth", [False, True], ids=["plain", "smoothquant"])
@pytest.mark.parametrize("name", ["downsample_conv", "resnet_conv"])
def test_w8a8_full_workloads_sampled(name, smooth):
    # the benchmark's workloads at full size, as the benchmark calls them (f32
    # out): sampled outputs and the four corners of every axis against the oracle
    wl = workloads.NAMED[name]()
    y = bt.bt_w8a8_conv2d(wl.x.to(DEV), wl.w.to(DEV), wl.stride, wl.padding, wl.dilation, smooth=smooth).cpu().numpy()
    rng = np.random.default_rng(3)
    idx = [rng.integers(0, n, 1500) for n in y.shape]
    corners = np.array(np.meshgrid(*[[0, n - 1] for n in y.shape], indexing="ij")).reshape(4, -1)
    b, o, i, j = [np.concatenate([a, c]) for a, c in zip(idx, corners)]
    flat = ((b * y.shape[1] + o) * y.shape[2] + i) * y.shape[3] + j
    want = oracle.w8a8_conv2d_at(wl.x.float().numpy(), wl.w.float().numpy(), wl.stride, wl.padding, wl.dilation,
                                 smooth, flat)
    np.testing.assert_array_equal(y.reshape(-1)[flat], want)
