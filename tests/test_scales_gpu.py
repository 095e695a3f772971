"""GPU: device-side scales. bt_scale_init against oracle.scale_init
(bit-exact for bf16 inputs, whose sum of |x| is exact in double on both
sides; within one fp32 step for f32 inputs), and the forward with device
scales against the same forward with host floats (bit-exact: both compute
alpha = fp32(scale_a * scale_w) from the same two floats)."""
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


@pytest.mark.parametrize("code", [bt.BT_CODE_BITS, bt.BT_CODE_E4M3, bt.BT_CODE_E2M1], ids=["bits", "e4m3", "e2m1"])
def test_linear_device_scales_equal_host_scales(code):
    x = torch.randn(300, 520, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).to(DEV)
    w = torch.randn(260, 520, generator=torch.Generator().manual_seed(2)).to(DEV)
    wp = bt.bt_pack_sign(w, code)
    sa = bt.bt_scale_init(x, 2.0)
    sw = torch.tensor([0.0123], dtype=torch.float32)
    scales = torch.cat([sa, sw.to(DEV)])
    host = bt.bt_binary_linear(x, wp, code, 520, float(sa.cpu()), float(sw), out_dtype=torch.float32)
    dev = bt.bt_binary_linear(x, wp, code, 520, scales, None, out_dtype=torch.float32)
    assert torch.equal(host.cpu(), dev.cpu())


@pytest.mark.parametrize("code", [bt.BT_CODE_BITS, bt.BT_CODE_E4M3, bt.BT_CODE_E2M1], ids=["bits", "e4m3", "e2m1"])
@pytest.mark.parametrize("s,p,d", [(1, 1, 1), (2, 1, 1), (2, 2, 2)])
def test_conv_device_scales_equal_host_scales(code, s, p, d):
    x = torch.randn(4, 64, 16, 16, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16).to(DEV)
    w = torch.randn(32, 64, 3, 3, generator=torch.Generator().manual_seed(4)).to(DEV)
    wp = bt.bt_pack_sign(w, code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    scales = torch.tensor([0.77, 0.031], dtype=torch.float32, device=DEV)
    host = bt.bt_binary_conv2d(x, wp, code, 64, 3, s, p, d, 0.77, 0.031)
    dev = bt.bt_binary_conv2d(x, wp, code, 64, 3, s, p, d, scales, None)
    assert torch.equal(host.cpu(), dev.cpu())
