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
