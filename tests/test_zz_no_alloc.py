"""bt_binary_linear_noalloc: the linear forward for callers that cannot
allocate device memory (it keeps the packed activations in the library's
fixed scratch array instead of a caller workspace).

Checked through the C ABI against bt_binary_linear, the entry point that takes
a workspace, on two calls in a row with different inputs, so that a second
call reading anything the first one left behind would show. This file is
collected last on purpose.
"""
import pytest
import torch

import xnor_popcount_gemm_gb300 as bt

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
REL_TOL = 1e-6


def _gen(seed, shape, dtype):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(dtype).to(DEV)


def _close(a, b):
    assert a.shape == b.shape and a.dtype == b.dtype
    if a.dtype == torch.int32:
        assert torch.equal(a, b)
    else:
        assert ((a.double() - b.double()).abs() <= REL_TOL * b.double().abs()).all()


@pytest.mark.parametrize("code", [bt.BT_CODE_BITS, bt.BT_CODE_E4M3, bt.BT_CODE_E2M1])
def test_noalloc_matches_workspace_entry_point_twice(code):
    K, N = 1000, 300
    w = _gen(1, (N, K), torch.bfloat16)
    wp = bt.bt_pack_sign(w, code)
    bias = torch.tensor([0.02], device=DEV)
    # second call: more rows, different data; the first call's scratch contents
    # must not leak into it
    for seed, M in ((2, 257), (3, 640)):
        x = _gen(seed, (M, K), torch.bfloat16)
        for od in (torch.int32, torch.bfloat16, torch.float32):
            want = bt.bt_binary_linear(x, wp, code, K, 0.8, 0.03, bias, out_dtype=od)
            got = bt.bt_binary_linear_noalloc(x, wp, code, K, 0.8, 0.03, bias, out_dtype=od)
            torch.cuda.synchronize()
            _close(got, want)
    assert bt.bt_device_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    cap = bt.bt_binary_linear_noalloc_max_bytes()
    K = 4096
    rows = cap // bt.bt_packed_row_bytes(K, bt.BT_CODE_E4M3) + 1
    x = torch.empty((rows, K), dtype=torch.bfloat16, device=DEV)
    wp = torch.empty((8, bt.bt_packed_row_bytes(K, bt.BT_CODE_E4M3)), dtype=torch.uint8, device=DEV)
    with pytest.raises(bt.BtError) as e:
        bt.bt_binary_linear_noalloc(x, wp, bt.BT_CODE_E4M3, K, 1.0, 1.0)
    assert e.value.status == bt.BT_ERR_WORKSPACE
