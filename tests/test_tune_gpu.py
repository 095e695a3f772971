"""The measured "ADAPTIVE" selection (bt_tune_linear, bt_plan): the tuning
call's own output and every later call in the shape it keeps give the
oracle's results bit for bit, the kept shape is the fastest it timed, and
bt_plan then names the fastest code measured for the size. (Each launch
shape on its own is checked against the oracle by the tile-configuration
tests of the parity suite.)"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads

import xnor_popcount_gemm_gb300 as bt

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TC_CODES = [bt.BT_CODE_E4M3, bt.BT_CODE_E2M1]


@pytest.fixture(autouse=True)
def _fresh_table():
    bt.bt_tune_reset()
    yield
    bt.bt_tune_reset()
    assert bt.bt_device_status() == 0


def _gen(seed, shape, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(dtype)


def _problem(M, N, K, dtype, seed=0):
    x = _gen(seed + M + K, (M, K), dtype)
    w = _gen(seed + N + 3 * K, (N, K), dtype)
    want = oracle.linear_dot(oracle.binarize(x), oracle.binarize_weight(w))
    return x, w, torch.from_numpy(want)


@pytest.mark.parametrize("code", TC_CODES, ids=["e4m3", "e2m1"])
@pytest.mark.parametrize("M,N,K", [(700, 600, 1000), (1100, 330, 4100), (2048, 1024, 2048)])
def test_tune_keeps_fastest_and_exact_shape(code, M, N, K):
    x, w, want = _problem(M, N, K, torch.bfloat16)
    xd, wp = x.to(DEV), bt.bt_pack_sign(w.to(DEV), code)
    out = torch.empty((M, N), dtype=torch.int32, device=DEV)
    res = bt.bt_tune_linear(xd, wp, code, K, 1.0, 1.0, out_dtype=torch.int32, reps=3, out=out)
    # the tuning call's own output (the last timed call) is the exact dot product
    assert torch.equal(out.cpu(), want)
    assert res["code"] == code and res["candidates"] >= 2
    assert res["us"] > 0.0 and res["us"] <= res["us_model"]
    assert res["epilogue_warps"] in (4, 8) and res["bn"] % 16 == 0 and 1 <= res["slices_per_stage"] <= 4
    # later calls of this size take the kept shape: still exact, scaled too
    got = bt.bt_binary_linear(xd, wp, code, K, 1.0, 1.0, out_dtype=torch.int32).cpu()
    assert torch.equal(got, want)
    sa, sw = workloads.mean_abs(x), workloads.mean_abs(w)
    y = bt.bt_binary_linear(xd, wp, code, K, sa, sw, out_dtype=torch.bfloat16).cpu()
    assert torch.equal(y, oracle.epilogue(want.numpy(), sa, sw, "bf16"))


@pytest.mark.parametrize("code", TC_CODES, ids=["e4m3", "e2m1"])
def test_tune_f32_input_with_bias(code):
    # f32 x with a per-feature shift: the tuning call's output (its last
    # candidate) and a later call (the kept shape) against the oracle
    M, K = 600, 1500
    for N in (480, 336, 200):
        x, w, _ = _problem(M, N, K, torch.float32, seed=N)
        xd, wp = x.to(DEV), bt.bt_pack_sign(w.to(DEV), code)
        bias = torch.linspace(-0.1, 0.1, K)
        want = torch.from_numpy(oracle.linear_dot(oracle.binarize(x, bias, channel_axis=-1),
                                                  oracle.binarize_weight(w)))
        out = torch.empty((M, N), dtype=torch.int32, device=DEV)
        res = bt.bt_tune_linear(xd, wp, code, K, 1.0, 1.0, bias_a=bias.to(DEV), out_dtype=torch.int32, reps=1,
                                out=out)
        assert torch.equal(out.cpu(), want)
        got = bt.bt_binary_linear(xd, wp, code, K, 1.0, 1.0, bias_a=bias.to(DEV), out_dtype=torch.int32).cpu()
        assert torch.equal(got, want), (N, res)


def test_plan_names_fastest_measured_code():
    M, N, K = 1024, 512, 3000
    x, w, want = _problem(M, N, K, torch.bfloat16)
    xd = x.to(DEV)
    before = bt.bt_plan(bt.BT_OP_LINEAR, M, N, K)
    times = {}
    for code in (bt.BT_CODE_BITS, bt.BT_CODE_E4M3, bt.BT_CODE_E2M1):
        wp = bt.bt_pack_sign(w.to(DEV), code)
        out = torch.empty((M, N), dtype=torch.int32, device=DEV)
        res = bt.bt_tune_linear(xd, wp, code, K, 1.0, 1.0, out_dtype=torch.int32, reps=3, out=out)
        assert torch.equal(out.cpu(), want)
        times[code] = res["us"]
    assert times[bt.BT_CODE_BITS] > 0
    code, algo = bt.bt_plan(bt.BT_OP_LINEAR, M, N, K)
    assert code == min(times, key=times.get)
    assert algo == {bt.BT_CODE_BITS: bt.BT_ALGO_POPC, bt.BT_CODE_E4M3: bt.BT_ALGO_TC_E4M3,
                    bt.BT_CODE_E2M1: bt.BT_ALGO_TC_E2M1}[code]
    # another size keeps the fixed rule; a reset forgets the measurement
    assert bt.bt_plan(bt.BT_OP_LINEAR, M + 1, N, K) == before
    bt.bt_tune_reset()
    assert bt.bt_plan(bt.BT_OP_LINEAR, M, N, K) == before


def test_tune_refuses_a_capturing_stream():
    M, N, K = 256, 256, 512
    x, w, _ = _problem(M, N, K, torch.bfloat16)
    code = bt.BT_CODE_E2M1
    xd, wp = x.to(DEV), bt.bt_pack_sign(w.to(DEV), code)
    out = torch.empty((M, N), dtype=torch.int32, device=DEV)
    ws = torch.empty(bt.bt_binary_linear_workspace(M, K, bt.BT_BF16, code), dtype=torch.uint8, device=DEV)
    res = bt.TuneResult()
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        st = bt._c_tune(xd.data_ptr(), bt.BT_BF16, wp.data_ptr(), code, M, N, K, 1.0, 1.0, None, 0,
                        out.data_ptr(), bt.BT_I32, ws.data_ptr(), ws.numel(), 3, s.cuda_stream, ctypes.byref(res))
    torch.cuda.synchronize()
    assert st == bt.BT_ERR_UNSUPPORTED
    # nothing was kept: the model's own shape still runs, exactly
    got = bt.bt_binary_linear(xd, wp, code, K, 1.0, 1.0, out_dtype=torch.int32).cpu()
    want = oracle.linear_dot(oracle.binarize(x), oracle.binarize_weight(w))
    np.testing.assert_array_equal(got.numpy(), want)
