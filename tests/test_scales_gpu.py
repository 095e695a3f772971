"""GPU: device-side scales. bt_scale_init against oracle.scale_init
(bit-exact for bf16 inputs, whose sum of |x| is exact in double on both
sides; within one fp32 step for f32 inputs), and the forwards that read the
scales from device memory against the oracle's whole forward called with the
oracle's own first-call scale (outputs within 1e-6 relative)."""
import numpy as np
import pytest
import torch

import oracle
import xnor_popcount_gemm_gb300 as bt

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _device_clean():
    yield
    assert bt.bt_device_status() == 0


@pytest.mark.parametrize("n", [1, 7, 1000, 123457, 4 * 1024 * 1024])
@pytest.mark.parametrize("dt,sdt", [(torch.bfloat16, torch.bfloat16), (torch.float32, torch.float32),
                                    (torch.bfloat16, torch.float32), (torch.float16, torch.float16)])
@pytest.mark.parametrize("factor", [2.0, 4.0])
def test_scale_init_matches_oracle(n, dt, sdt, factor):
    x = torch.randn(n, generator=torch.Generator().manual_seed(n)).to(dt)
    got = float(bt.bt_scale_init(x.to(DEV), factor, sdt).cpu())
    names = {torch.bfloat16: "bf16", torch.float32: "f32", torch.float16: "f16"}
    want = oracle.scale_init(x.float().numpy(), factor, names[dt], names[sdt])
    if dt == torch.float32:
        assert abs(got - want) <= abs(want) * 2.0 ** -23
    else:
        assert got == want


CODES = [bt.BT_CODE_BITS, bt.BT_CODE_E4M3, bt.BT_CODE_E2M1]
CODE_IDS = ["bits", "e4m3", "e2m1"]


def _close_rel(got, want):
    assert got.shape == want.shape and got.dtype == want.dtype
    assert ((got.double() - want.double()).abs() <= 1e-6 * want.double().abs()).all()


@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
@pytest.mark.parametrize("od", ["f32", "bf16"])
def test_linear_device_scales_match_oracle(code, od):
    # first-call scale from x on the device (factor 2, bf16 x, bf16 scale as
    # set_activation keeps it in the layer dtype), scale_w a device float;
    # expected: the oracle's scale_init and its whole forward with that scale
    x = torch.randn(300, 520, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    w = torch.randn(260, 520, generator=torch.Generator().manual_seed(2))
    bias = torch.tensor([-0.03])
    wp = bt.bt_pack_sign(w.to(DEV), code)
    sa = bt.bt_scale_init(x.to(DEV), 2.0, torch.bfloat16)
    sw = torch.tensor([0.0123], dtype=torch.float32)
    scales = torch.cat([sa.float(), sw.to(DEV)])
    want_sa = oracle.scale_init(x.float().numpy(), 2.0, "bf16", "bf16")
    assert float(sa.cpu()) == want_sa
    out_t = {"f32": torch.float32, "bf16": torch.bfloat16}[od]
    got = bt.bt_binary_linear(x.to(DEV), wp, code, 520, scales, None, bias.to(DEV), out_dtype=out_t).cpu()
    want = oracle.binary_linear(x, w, want_sa, float(sw), bias, od)
    _close_rel(got, want)


@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
@pytest.mark.parametrize("s,p,d", [(1, 1, 1), (2, 1, 1), (2, 2, 2)])
def test_conv_device_scales_match_oracle(code, s, p, d):
    x = torch.randn(4, 64, 16, 16, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    w = torch.randn(32, 64, 3, 3, generator=torch.Generator().manual_seed(4))
    bias = torch.linspace(-0.1, 0.1, 64)
    wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    sa = bt.bt_scale_init(x.to(DEV), 4.0, torch.float32)
    scales = torch.cat([sa, torch.tensor([0.031], device=DEV)])
    want_sa = oracle.scale_init(x.float().numpy(), 4.0, "bf16", "f32")
    assert float(sa.cpu()) == want_sa
    got = bt.bt_binary_conv2d(x.to(DEV), wp, code, 64, 3, s, p, d, scales, None, bias.to(DEV)).cpu()
    want = oracle.binary_conv2d(x, w, want_sa, 0.031, s, p, d, bias, "bf16")
    _close_rel(got, want)


# ---------------------------------------------------------------------------
# A layer's first forward: scale_a computed from the read of x that packs it
# (bt_binary_*_dscale_init), then the forward with it.
# ---------------------------------------------------------------------------

NAMES = {torch.bfloat16: "bf16", torch.float32: "f32", torch.float16: "f16"}


def _check_scale(got, want, x_dtype):
    # bf16 / f16 x: the rounded mean equals the oracle's for these inputs; f32
    # x: within the sum's error (a few units of 2^-24 relative)
    if x_dtype == torch.float32:
        assert abs(got - want) <= abs(want) * 4 * 2.0 ** -24
    else:
        assert got == want


@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32, torch.float16])
@pytest.mark.parametrize("M,K", [(300, 520), (257, 1001), (64, 4096)])
def test_linear_first_forward_scale_and_output(code, dt, M, K):
    # K = 1001 (rows not 8-byte aligned) takes the two-pass fallback
    x = torch.randn(M, K, generator=torch.Generator().manual_seed(M + K)).to(dt)
    w = torch.randn(129, K, generator=torch.Generator().manual_seed(7))
    bias = torch.tensor([0.05])
    wp = bt.bt_pack_sign(w.to(DEV), code)
    scales = torch.tensor([0.0, 0.021], dtype=torch.float32, device=DEV)
    for factor, sdt in ((2.0, dt), (4.0, torch.float32)):
        got = bt.bt_binary_linear_dscale_init(x.to(DEV), wp, code, K, scales, factor, sdt, bias.to(DEV),
                                              out_dtype=torch.float32).cpu()
        sa = float(scales[0].cpu())
        want_sa = oracle.scale_init(x.float().numpy(), factor, NAMES[dt], NAMES[sdt])
        _check_scale(sa, want_sa, dt)
        _close_rel(got, oracle.binary_linear(x, w, sa, 0.021, bias, "f32"))


@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,C,H,W,s,p,d", [(4, 64, 16, 16, 1, 1, 1), (3, 128, 28, 28, 2, 1, 1),
                                           (2, 40, 7, 9, 2, 2, 2), (1, 16, 3, 300, 1, 1, 1)])
def test_conv_first_forward_scale_and_output(code, dt, B, C, H, W, s, p, d):
    # 7 x 9 planes (not 16-byte aligned) take the two-pass fallback; 300-wide
    # rows the explicit unfold
    x = torch.randn(B, C, H, W, generator=torch.Generator().manual_seed(B * C + H)).to(dt)
    w = torch.randn(33, C, 3, 3, generator=torch.Generator().manual_seed(9))
    bias = torch.linspace(-0.1, 0.1, C)
    wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    scales = torch.tensor([0.0, 0.031], dtype=torch.float32, device=DEV)
    got = bt.bt_binary_conv2d_dscale_init(x.to(DEV), wp, code, 3, s, p, d, scales, 2.0, None, bias.to(DEV)).cpu()
    sa = float(scales[0].cpu())
    want_sa = oracle.scale_init(x.float().numpy(), 2.0, NAMES[dt], NAMES[dt])
    _check_scale(sa, want_sa, dt)
    _close_rel(got, oracle.binary_conv2d(x, w, sa, 0.031, s, p, d, bias, NAMES[dt]))
