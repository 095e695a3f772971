"""bt_binary_linear_noalloc: the linear forward for callers that cannot
allocate device memory -- code inside a host framework that owns every device
allocation (a plugin's enqueue callback, say), or under a fixed memory budget.
It keeps the packed activations in the library's fixed scratch array instead
of a caller workspace.

Checked through the C ABI against the CPU oracle (integer outputs bit for bit,
scaled outputs within 1e-6 relative) and against bt_binary_linear, the entry
point that takes a workspace, on two calls in a row with different inputs, so
that a second call reading anything the first one left behind would show. Also:
packed activations into a caller's output tensor, the largest problem the
scratch holds, the refusal one row past it, and that a call changes neither
torch's allocation count nor the device's free memory. This file is collected
last on purpose.
"""
import gc

import numpy as np
import pytest
import torch

import oracle
import xnor_popcount_gemm_gb300 as bt

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
REL_TOL = 1e-6
CODES = [bt.BT_CODE_BITS, bt.BT_CODE_E4M3, bt.BT_CODE_E2M1]
CODE_IDS = ["bits", "e4m3", "e2m1"]
OUT_NAME = {torch.int32: "i32", torch.bfloat16: "bf16", torch.float32: "f32"}


def _gen(seed, shape, dtype):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(dtype)


def _close(got, want):
    assert got.shape == want.shape and got.dtype == want.dtype
    if got.dtype == torch.int32:
        assert torch.equal(got, want)
    else:
        assert ((got.double() - want.double()).abs() <= REL_TOL * want.double().abs()).all()


@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(code):
    K, N = 1000, 300
    w = _gen(1, (N, K), torch.bfloat16)
    wp = bt.bt_pack_sign(w.to(DEV), code)
    bias = torch.tensor([0.02])
    sw = oracle.binarize_weight(w)
    # second call: more rows, different data; the first call's scratch contents
    # must not leak into it
    for seed, M in ((2, 257), (3, 640)):
        x = _gen(seed, (M, K), torch.bfloat16)
        want_dot = oracle.linear_dot(oracle.binarize(x, bias, channel_axis=-1), sw)
        xd = x.to(DEV)
        for od in (torch.int32, torch.bfloat16, torch.float32):
            got = bt.bt_binary_linear_noalloc(xd, wp, code, K, 0.8, 0.03, bias.to(DEV), out_dtype=od)
            ref = bt.bt_binary_linear(xd, wp, code, K, 0.8, 0.03, bias.to(DEV), out_dtype=od)
            torch.cuda.synchronize()
            _close(got.cpu(), oracle.epilogue(want_dot, 0.8, 0.03, OUT_NAME[od]))
            _close(got.cpu(), ref.cpu())
    assert bt.bt_device_status() == 0


@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
def test_noalloc_packed_input_into_callers_output(code):
    M, N, K = 300, 130, 777
    x = _gen(4, (M, K), torch.float32)
    w = _gen(5, (N, K), torch.float32)
    xp = bt.bt_pack_sign(x.to(DEV), code)
    wp = bt.bt_pack_sign(w.to(DEV), code)
    out = torch.full((M, N), -7, dtype=torch.int32, device=DEV)
    got = bt.bt_binary_linear_noalloc(xp, wp, code, K, 1.0, 1.0, out_dtype=torch.int32, x_packed=True, out=out)
    assert got.data_ptr() == out.data_ptr()
    want = oracle.linear_dot(oracle.binarize(x), oracle.binarize_weight(w))
    assert np.array_equal(out.cpu().numpy(), want)
    assert bt.bt_device_status() == 0


@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
def test_noalloc_largest_problem_the_scratch_holds(code):
    cap = bt.bt_binary_linear_noalloc_max_bytes()
    K, N = 4096, 40
    M = cap // bt.bt_packed_row_bytes(K, code)
    assert bt.bt_binary_linear_workspace(M, K, bt.BT_BF16, code) <= cap
    x = _gen(6, (M, K), torch.bfloat16)
    w = _gen(7, (N, K), torch.bfloat16)
    wp = bt.bt_pack_sign(w.to(DEV), code)
    got = bt.bt_binary_linear_noalloc(x.to(DEV), wp, code, K, 1.0, 1.0, out_dtype=torch.int32)
    want = oracle.linear_dot(oracle.binarize(x), oracle.binarize_weight(w))
    assert np.array_equal(got.cpu().numpy(), want)
    # one row more does not fit
    xd = torch.empty((M + 1, K), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(bt.BtError) as e:
        bt.bt_binary_linear_noalloc(xd, wp, code, K, 1.0, 1.0, out_dtype=torch.int32)
    assert e.value.status == bt.BT_ERR_WORKSPACE
    assert bt.bt_device_status() == 0


def test_noalloc_allocates_nothing():
    code = bt.BT_CODE_E2M1
    M, N, K = 512, 256, 2048
    x = _gen(8, (M, K), torch.bfloat16).to(DEV)
    wp = bt.bt_pack_sign(_gen(9, (N, K), torch.bfloat16).to(DEV), code)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    # the first call may load the library's module (and with it the array)
    bt.bt_binary_linear_noalloc(x, wp, code, K, 1.0, 1.0, out=out)
    torch.cuda.synchronize()
    # tensors that earlier tests left in reference cycles are freed now, and no
    # collection runs inside the window (it would lower the count, not raise it)
    gc.collect()
    gc.disable()
    try:
        used0 = torch.cuda.memory_allocated()
        free0, _ = torch.cuda.mem_get_info()
        for _ in range(3):
            bt.bt_binary_linear_noalloc(x, wp, code, K, 1.0, 1.0, out=out)
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        used1 = torch.cuda.memory_allocated()
    finally:
        gc.enable()
    assert used1 == used0
    assert free1 == free0
    assert bt.bt_device_status() == 0
