"""GPU: the bounded-wait timeout path, exercised without breaking anything.

bt_set_wait_timeout(1) makes every bounded wait of the tensor-core kernels'
main loops give up after 1 ns, i.e. at the first wait that has to wait at all
(a copy or an MMA in flight). The kernel then records BT_ERR_TIMEOUT in the
device error word, lets its copies and MMAs in flight finish (those drains
keep the 2 s limit), frees its tensor memory and returns. The test checks that
bt_device_status reports the timeout once, and that the next call at the
default limit is bit-exact against the oracle on the same, still usable,
context. Covered: single-CTA and CTA-pair linear tiles, the implicit-im2col
convolution.
"""
import numpy as np
import pytest
import torch

import oracle
import xnor_popcount_gemm_gb300 as bt

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _gen(seed, shape):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16)


def _timed_out(call):
    assert bt.bt_device_status() == 0
    bt.bt_set_wait_timeout(1)
    try:
        call()
        status = bt.bt_device_status()
    finally:
        bt.bt_set_wait_timeout(0)
    return status


@pytest.mark.parametrize("cfg", ["128,1", "pair,128,2"])
def test_linear_wait_timeout_reports_and_recovers(cfg, monkeypatch):
    monkeypatch.setenv("BT_TC_CONFIG", cfg)
    code = bt.BT_CODE_E2M1
    M, N, K = 700, 600, 2048
    x, w = _gen(1, (M, K)), _gen(2, (N, K))
    xd = x.to(DEV)
    wp = bt.bt_pack_sign(w.to(DEV), code)
    status = _timed_out(lambda: bt.bt_binary_linear(xd, wp, code, K, 1.0, 1.0, out_dtype=torch.int32))
    assert status == bt.BT_ERR_TIMEOUT
    assert bt.bt_device_status() == 0          # reported once, then cleared
    got = bt.bt_binary_linear(xd, wp, code, K, 1.0, 1.0, out_dtype=torch.int32).cpu()
    want = oracle.linear_dot(oracle.binarize(x), oracle.binarize_weight(w))
    assert np.array_equal(got.numpy(), want)
    assert bt.bt_device_status() == 0


def test_conv_wait_timeout_reports_and_recovers():
    code = bt.BT_CODE_E2M1
    B, C, H, W, O, k, s, p, d = 4, 128, 28, 28, 256, 3, 2, 1, 1
    x, w = _gen(3, (B, C, H, W)), _gen(4, (O, C, k, k))
    xd = x.to(DEV)
    wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    run = lambda: bt.bt_binary_conv2d(xd, wp, code, C, k, s, p, d, 1.0, 1.0, out_dtype=torch.int32)
    assert _timed_out(run) == bt.BT_ERR_TIMEOUT
    got = run().cpu()
    want = oracle.conv2d_dot(oracle.binarize(x), oracle.binarize_weight(w), s, p, d)
    assert np.array_equal(got.numpy(), want)
    assert bt.bt_device_status() == 0
