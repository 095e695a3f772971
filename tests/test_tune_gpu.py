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


# ---------------------------------------------------------------------------
# Convolution: the implicit plans (pairs or single CTAs, resident or streamed
# weights, one or two pixel stages, with or without the convolution packing x
# itself)
# ---------------------------------------------------------------------------

CONV_GEOMS = [  # B, C, H, W, O, k, s, p, d, x dtype
    (2, 128, 28, 28, 256, 3, 2, 1, 1, torch.bfloat16),
    (2, 128, 28, 28, 256, 3, 2, 2, 2, torch.bfloat16),
    (2, 256, 14, 14, 256, 3, 1, 1, 1, torch.float32),
    (3, 64, 17, 19, 96, 3, 1, 1, 1, torch.float32),
]


@pytest.mark.parametrize("code", TC_CODES, ids=["e4m3", "e2m1"])
@pytest.mark.parametrize("geom", CONV_GEOMS, ids=["s2p1", "s2p2d2", "s1p1", "ragged"])
def test_tune_conv_keeps_fastest_and_exact_plan(code, geom):
    B, C, H, W, O, k, s, p, d, dt = geom
    x = _gen(B + C + H, (B, C, H, W), dt)
    w = _gen(O + C, (O, C, k, k), dt)
    want = torch.from_numpy(oracle.conv2d_dot(oracle.binarize(x), oracle.binarize_weight(w), s, p, d))
    xd, wp = x.to(DEV), bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    out = torch.empty(want.shape, dtype=torch.int32, device=DEV)
    res = bt.bt_tune_conv2d(xd, wp, code, C, k, s, p, d, 1.0, 1.0, out_dtype=torch.int32, reps=2, out=out)
    assert torch.equal(out.cpu(), want)
    assert res["code"] == code and res["candidates"] >= (2 if O > 128 else 1)
    assert res["us"] > 0.0 and res["us"] <= res["us_model"]
    assert res["pixel_stages"] in (1, 2) and res["pair"] in (0, 1) and res["fused"] in (0, 1)
    # later calls of the geometry take the kept plan: on x, and on packed pixels
    got = bt.bt_binary_conv2d(xd, wp, code, C, k, s, p, d, 1.0, 1.0, out_dtype=torch.int32).cpu()
    assert torch.equal(got, want)
    xp = bt.bt_pack_sign(xd, code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    got = bt.bt_binary_conv2d(xp, wp, code, C, k, s, p, d, 1.0, 1.0, out_dtype=torch.int32, x_packed=True).cpu()
    assert torch.equal(got, want)
    sa, sw = workloads.mean_abs(x), workloads.mean_abs(w)
    ot = "bf16" if dt == torch.bfloat16 else "f32"
    y = bt.bt_binary_conv2d(xd, wp, code, C, k, s, p, d, sa, sw).cpu()
    assert torch.equal(y, oracle.epilogue(want.numpy(), sa, sw, ot))
    # the split the library reports for the geometry follows the kept route
    xt = {torch.float32: bt.BT_F32, torch.bfloat16: bt.BT_BF16}[dt]
    mode = bt.bt_conv2d_single_pass(B, C, H, W, k, s, p, d, xt, code)
    assert (mode == 2) == (res["fused"] == 1)


def test_plan_names_fastest_measured_conv_code():
    B, C, H, W, O, k, s, p, d = 2, 128, 28, 28, 256, 3, 2, 1, 1
    x = _gen(5, (B, C, H, W), torch.bfloat16)
    w = _gen(6, (O, C, k, k), torch.bfloat16)
    want = torch.from_numpy(oracle.conv2d_dot(oracle.binarize(x), oracle.binarize_weight(w), s, p, d))
    Ho = bt.conv2d_out_size(H, k, s, p, d)
    M, N, K = B * Ho * Ho, O, C * k * k
    before = bt.bt_plan(bt.BT_OP_CONV2D, M, N, K)
    times = {}
    for code in (bt.BT_CODE_BITS, bt.BT_CODE_E4M3, bt.BT_CODE_E2M1):
        wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
        out = torch.empty(want.shape, dtype=torch.int32, device=DEV)
        res = bt.bt_tune_conv2d(x.to(DEV), wp, code, C, k, s, p, d, 1.0, 1.0, out_dtype=torch.int32, reps=2,
                                out=out)
        assert torch.equal(out.cpu(), want)
        times[code] = res["us"]
    assert bt.bt_plan(bt.BT_OP_CONV2D, M, N, K)[0] == min(times, key=times.get)
    bt.bt_tune_reset()
    assert bt.bt_plan(bt.BT_OP_CONV2D, M, N, K) == before


# ---------------------------------------------------------------------------
# BT_ALGO_TUNE: the forward entry points tune a size on its first call
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("code", TC_CODES, ids=["e4m3", "e2m1"])
def test_algo_tune_linear_first_call_tunes(code):
    M, N, K = 900, 520, 1700
    x, w, want = _problem(M, N, K, torch.bfloat16, seed=7)
    xd, wp = x.to(DEV), bt.bt_pack_sign(w.to(DEV), code)
    for _ in range(2):          # the first call tunes, the second takes the kept shape
        got = bt.bt_binary_linear(xd, wp, code, K, 1.0, 1.0, out_dtype=torch.int32, algo=bt.BT_ALGO_TUNE).cpu()
        assert torch.equal(got, want)
    # the size was timed: bt_plan names the one code measured for it
    assert bt.bt_plan(bt.BT_OP_LINEAR, M, N, K)[0] == code


@pytest.mark.parametrize("code", TC_CODES, ids=["e4m3", "e2m1"])
def test_algo_tune_conv_first_call_tunes(code):
    B, C, H, W, O, k, s, p, d = 2, 128, 28, 28, 256, 3, 2, 1, 1
    x = _gen(11, (B, C, H, W), torch.bfloat16)
    w = _gen(12, (O, C, k, k), torch.bfloat16)
    want = torch.from_numpy(oracle.conv2d_dot(oracle.binarize(x), oracle.binarize_weight(w), s, p, d))
    xd, wp = x.to(DEV), bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    for _ in range(2):
        got = bt.bt_binary_conv2d(xd, wp, code, C, k, s, p, d, 1.0, 1.0, out_dtype=torch.int32,
                                  algo=bt.BT_ALGO_TUNE).cpu()
        assert torch.equal(got, want)
    Ho = bt.conv2d_out_size(H, k, s, p, d)
    assert bt.bt_plan(bt.BT_OP_CONV2D, B * Ho * Ho, O, C * k * k)[0] == code


def test_algo_tune_inside_a_capture_runs_as_auto():
    M, N, K = 512, 384, 1000
    code = bt.BT_CODE_E4M3
    x, w, want = _problem(M, N, K, torch.bfloat16, seed=9)
    xd, wp = x.to(DEV), bt.bt_pack_sign(w.to(DEV), code)
    out = torch.empty((M, N), dtype=torch.int32, device=DEV)
    ws = torch.empty(bt.bt_binary_linear_workspace(M, K, bt.BT_BF16, code), dtype=torch.uint8, device=DEV)
    before = bt.bt_plan(bt.BT_OP_LINEAR, M, N, K)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        bt.bt_binary_linear(xd, wp, code, K, 1.0, 1.0, out_dtype=torch.int32, algo=bt.BT_ALGO_TUNE, out=out,
                            workspace=ws)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), want)
    # nothing was timed or kept
    assert bt.bt_plan(bt.BT_OP_LINEAR, M, N, K) == before
