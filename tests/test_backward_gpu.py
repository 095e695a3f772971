"""GPU parity of the straight-through backward of the binary linear layer
(bt_sign_transpose + bt_binary_linear_backward, through the C ABI) against
oracle.linear_backward.

The tensor cores accumulate exact bf16 products in fp32, the oracle sums
them exactly (float64); each side rounds its sum once to bf16. So an output
may differ from the oracle's by the fp32 accumulation error, which can move
the bf16 rounding by one step: every output must lie within
max(one bf16 step of the oracle's value, n * 2^-23 * sum_j |terms_j|) of the
oracle's, n the contraction length (the classical bound n*u*sum|terms| for a
sum of n floats with unit roundoff u = 2^-24, doubled for the scale). The
straight-through mask is an integer decision taken in x's dtype on both sides
and must agree exactly; grad_scale_a (fp32 terms, summed in no fixed order
on the GPU) must lie within 1e-5 of the sum of |terms| plus the terms of the
outputs where the two grad_inputs differ.
"""
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


def _inputs(M, N, K, x_dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    x = torch.randn(M, K, generator=gen).to(x_dtype)
    w = (torch.randn(N, K, generator=gen) * 0.02).to(torch.bfloat16)
    g = (torch.randn(M, N, generator=gen) * 0.01).to(torch.bfloat16)
    x.view(-1)[:4] = torch.tensor([0.0, -0.0, 1e-30, -1e-30]).to(x_dtype)[: min(4, x.numel())]
    w.view(-1)[0] = 0.0
    scale_a = float(x.float().abs().mean())
    scale_w = float(w.float().abs().mean())
    return x, w, g, scale_a, scale_w


def _bf16_step(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |v| (2^(e-7) for |v| in [2^e, 2^(e+1)))."""
    a = np.abs(v.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def _check_sum(got, want, abs_terms, n, what):
    got = got.astype(np.float64)
    tol = np.maximum(_bf16_step(want), n * 2.0 ** -23 * abs_terms)
    bad = np.abs(got - want.astype(np.float64)) > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside tolerance, first {np.argwhere(bad)[0].tolist()}"


def _run(M, N, K, x_dtype, gw_dtype, seed=0):
    x, w, g, sa, sw = _inputs(M, N, K, x_dtype, seed)
    wst = bt.bt_sign_transpose(w.to(DEV))
    gx, gsa, gw = bt.bt_binary_linear_backward(x.to(DEV), wst, g.to(DEV), sa, sw, grad_weight_dtype=gw_dtype)
    torch.cuda.synchronize()
    return x, w, g, sa, sw, gx.cpu(), float(gsa.cpu()), gw.cpu()


def _compare(x, w, g, sa, sw, gx, gsa, gw, x_dt):
    o = oracle.linear_backward(x.float().numpy(), w.float().numpy(), g.float().numpy(), sa, sw, x_dt)
    g64 = g.double().numpy()
    bw = float(oracle.bf16_round(np.float32(sw)))
    ba = float(oracle.bf16_round(np.float32(sa)))
    M, K = x.shape
    N = w.shape[0]
    # grad_input: mask exactly, values within the bound
    gxn = gx.float().numpy()
    masked = o["middle"] == 0
    assert np.all(gxn[masked] == 0), "mask disagrees"
    abs_in = np.abs(g64).sum(1, keepdims=True) * bw * np.ones((1, K))
    _check_sum(gxn, o["grad_input"], abs_in, N, "grad_input")
    # grad_scale_a
    differ = gxn != o["grad_input"]
    extra = float(np.abs(o["grad_input"][differ]).sum()) / np.sqrt(M * K) * 2.0 ** -7
    assert abs(gsa - o["grad_scale_a"]) <= 1e-5 * o["grad_scale_a_abs"] + extra + 1e-30, (gsa, o["grad_scale_a"])
    # grad_weight
    abs_w = np.abs(g64).sum(0)[:, None] * ba * np.ones((1, K))
    if gw.dtype == torch.bfloat16:
        _check_sum(gw.float().numpy(), o["grad_weight"], abs_w, M, "grad_weight")
    else:
        got = gw.double().numpy()
        bad = np.abs(got - o["grad_weight_exact"]) > M * 2.0 ** -23 * abs_w + 1e-30
        assert not bad.any(), f"grad_weight f32: {int(bad.sum())} outside the fp32 bound"
    return o, differ


SHAPES = [(64, 64, 64), (128, 8, 16), (200, 136, 264), (333, 520, 72), (1000, 264, 1040), (257, 1024, 512)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("x_dtype", [torch.bfloat16, torch.float32], ids=["x_bf16", "x_f32"])
def test_linear_backward_matches_oracle(M, N, K, x_dtype):
    x, w, g, sa, sw, gx, gsa, gw = _run(M, N, K, x_dtype, torch.bfloat16, seed=M + N + K)
    _, differ = _compare(x, w, g, sa, sw, gx, gsa, gw, "bf16" if x_dtype == torch.bfloat16 else "f32")
    assert differ.mean() < 0.01                  # almost every bf16 output is the exact one


@pytest.mark.parametrize("M,N,K", [(200, 136, 264), (1000, 264, 1040)])
def test_linear_backward_grad_weight_f32(M, N, K):
    x, w, g, sa, sw, gx, gsa, gw = _run(M, N, K, torch.bfloat16, torch.float32, seed=7)
    _compare(x, w, g, sa, sw, gx, gsa, gw, "bf16")


def test_linear_backward_mask_decided_in_x_dtype():
    # x / scale_a just above 1: masked for an f32 x, kept for a bf16 x (the
    # quotient rounds to exactly 1.0 in bf16)
    M, N, K = 128, 64, 64
    sa = 0.998046875
    x = torch.full((M, K), 1.0)
    w = torch.ones(N, K, dtype=torch.bfloat16)
    g = torch.ones(M, N, dtype=torch.bfloat16)
    wst = bt.bt_sign_transpose(w.to(DEV))
    gx16, _, _ = bt.bt_binary_linear_backward(x.to(torch.bfloat16).to(DEV), wst, g.to(DEV), sa, 1.0,
                                             grad_weight_dtype=None)
    gx32, _, _ = bt.bt_binary_linear_backward(x.to(DEV), wst, g.to(DEV), sa, 1.0, grad_weight_dtype=None)
    assert torch.all(gx16.cpu().float() == float(N)) and torch.all(gx32.cpu().float() == 0.0)


def test_linear_backward_sign_transpose():
    w = torch.randn(300, 136).to(torch.bfloat16)
    w[0, :3] = torch.tensor([0.0, -0.0, float("nan")]).to(torch.bfloat16)
    got = bt.bt_sign_transpose(w.to(DEV)).cpu()
    assert got.shape == (136, bt.bt_backward_weight_ld(300)) == (136, 320)
    want = torch.zeros(136, 320, dtype=torch.bfloat16)
    want[:, :300] = w.float().sign().t().to(torch.bfloat16)
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    got32 = bt.bt_sign_transpose(w.float().to(DEV), ld=304).cpu()
    assert torch.equal(got32[:, :300], want[:, :300]) and torch.all(got32[:, 300:] == 0)


@pytest.mark.parametrize("R,C,dtype", [(300, 136, torch.float16), (77, 13, torch.bfloat16), (1030, 72, torch.float32),
                                       (9, 8, torch.float16), (513, 264, torch.bfloat16)])
def test_sign_transpose_shapes_and_special_values(R, C, dtype):
    w = torch.randn(R, C, generator=torch.Generator().manual_seed(R * C)).to(dtype)
    specials = torch.tensor([0.0, -0.0, float("nan"), float("inf"), -float("inf"), -1e-3, 1e-3])
    w.view(-1)[: specials.numel()] = specials.to(dtype)[: w.numel()]
    ld = bt.bt_backward_weight_ld(R)
    got = bt.bt_sign_transpose(w.to(DEV)).cpu()
    want = torch.zeros(C, ld, dtype=torch.bfloat16)
    want[:, :R] = torch.from_numpy(oracle.sign(w.float().numpy())).t().to(torch.bfloat16)
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_linear_backward_partial_requests_and_empty():
    x, w, g, sa, sw = _inputs(130, 64, 96, torch.bfloat16, 3)
    wst = bt.bt_sign_transpose(w.to(DEV))
    gx, gsa, gw = bt.bt_binary_linear_backward(x.to(DEV), wst, g.to(DEV), sa, sw, grad_weight_dtype=None)
    assert gw is None and gx is not None
    gx2, gsa2, gw2 = bt.bt_binary_linear_backward(x.to(DEV), None, g.to(DEV), sa, sw, grad_input=False)
    assert gx2 is None and gsa2 is None and gw2 is not None
    gx3, gsa3, gw3 = bt.bt_binary_linear_backward(x.to(DEV), wst, g.to(DEV), sa, sw)
    assert torch.equal(gx3.cpu(), gx.cpu()) and torch.equal(gw3.cpu(), gw2.cpu())
    e = torch.empty(0, 96, dtype=torch.bfloat16, device=DEV)
    ge = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    gxe, gsae, gwe = bt.bt_binary_linear_backward(e, wst, ge, sa, sw)
    assert gxe.numel() == 0 and float(gsae.cpu()) == 0.0 and torch.all(gwe.cpu() == 0)


@pytest.mark.parametrize("epi", ["4", "8"], ids=["epi4", "epi8"])
@pytest.mark.parametrize("cfg", ["pair,224,2", "pair,128,2", "224,2", "128,4", "64,1", "pair,256,1"])
def test_linear_backward_tile_configs(cfg, epi, monkeypatch):
    # epi: one or two epilogue warps per TMEM lane quarter (the masked layouts
    # run two unless forced)
    monkeypatch.setenv("BT_TC_CONFIG", cfg)
    monkeypatch.setenv("BT_TC_EPI", epi)
    x, w, g, sa, sw, gx, gsa, gw = _run(300, 264, 520, torch.bfloat16, torch.bfloat16, seed=11)
    _compare(x, w, g, sa, sw, gx, gsa, gw, "bf16")


@pytest.mark.slow
def test_linear_backward_full_size_sampled():
    # the 4096 x 4096 x 4096 bf16 layer: the oracle computes sampled rows of
    # grad_input and sampled rows of grad_weight
    M = N = K = 4096
    x, w, g, sa, sw = _inputs(M, N, K, torch.bfloat16, 2)
    wst = bt.bt_sign_transpose(w.to(DEV))
    gx, gsa, gw = bt.bt_binary_linear_backward(x.to(DEV), wst, g.to(DEV), sa, sw)
    torch.cuda.synchronize()
    gx, gw = gx.cpu(), gw.cpu()
    rows = np.array([0, 1, 127, 128, 2047, 4000, 4095])
    o = oracle.linear_backward(x[rows].float().numpy(), w.float().numpy(), g[rows].float().numpy(), sa, sw, "bf16")
    g64 = g.double().numpy()
    bw = float(oracle.bf16_round(np.float32(sw)))
    _check_sum(gx[rows].float().numpy(), o["grad_input"], np.abs(g64[rows]).sum(1, keepdims=True) * bw * np.ones((1, K)),
               N, "grad_input rows")
    assert np.all(gx[rows].float().numpy()[o["middle"] == 0] == 0)
    cols = np.array([0, 5, 255, 256, 3071, 4095])
    xs = oracle.bf16_round(oracle.sign(x.float().numpy()) * np.float32(sa)).astype(np.float64)
    gw_exact = g64[:, cols].T @ xs
    ba = float(oracle.bf16_round(np.float32(sa)))
    _check_sum(gw[cols].float().numpy(), oracle.bf16_round(gw_exact), np.abs(g64[:, cols]).sum(0)[:, None] * ba * np.ones((1, K)),
               M, "grad_weight rows")
    # grad_scale_a over every output: recompute the terms from the GPU's own grad_input
    xf = x.float().numpy()
    terms = ((gx.float().numpy() * oracle.sign(xf)).astype(np.float32) * np.float32(1.0 / np.sqrt(M * K))).astype(np.float64)
    assert abs(float(gsa.cpu()) - terms.sum()) <= 1e-5 * np.abs(terms).sum()


# ---------------------------------------------------------------------------
# conv2d
# ---------------------------------------------------------------------------

def _conv_inputs(B, C, H, W, O, k, s, p, d, x_dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    Ho, Wo = oracle.conv2d_out_size(H, k, s, p, d), oracle.conv2d_out_size(W, k, s, p, d)
    x = torch.randn(B, C, H, W, generator=gen).to(x_dtype)
    w = (torch.randn(O, C, k, k, generator=gen) * 0.05).to(torch.bfloat16)
    g = (torch.randn(B, O, Ho, Wo, generator=gen) * 0.01).to(torch.bfloat16)
    x.view(-1)[:2] = torch.tensor([0.0, -0.0]).to(x_dtype)
    w.view(-1)[0] = 0.0
    return x, w, g, float(x.float().abs().mean()), float(w.float().abs().mean())


def _conv_run_and_compare(B, C, H, W, O, k, s, p, d, x_dtype, gw_dtype, seed):
    x, w, g, sa, sw = _conv_inputs(B, C, H, W, O, k, s, p, d, x_dtype, seed)
    wst = bt.bt_sign_transpose(w.view(O, -1).to(DEV))
    gx, gsa, gw = bt.bt_binary_conv2d_backward(x.to(DEV), wst, g.to(DEV), O, k, s, p, d, sa, sw,
                                               grad_weight_dtype=gw_dtype)
    torch.cuda.synchronize()
    gx, gsa, gw = gx.cpu(), float(gsa.cpu()), gw.cpu()
    x_dt = "bf16" if x_dtype == torch.bfloat16 else "f32"
    o = oracle.conv2d_backward(x.float().numpy(), w.float().numpy(), g.float().numpy(), sa, sw, s, p, d, x_dt)
    # per-output bounds from the same sums over absolute values
    ag = g.double().abs()
    bw = float(oracle.bf16_round(np.float32(sw)))
    ba = float(oracle.bf16_round(np.float32(sa)))
    abs_in = torch.nn.grad.conv2d_input(x.shape, torch.full(w.shape, bw, dtype=torch.float64), ag, stride=s,
                                        padding=p, dilation=d).numpy()
    abs_w = torch.nn.grad.conv2d_weight(torch.full(x.shape, ba, dtype=torch.float64), w.shape, ag, stride=s,
                                        padding=p, dilation=d).numpy()
    gxn = gx.float().numpy()
    assert np.all(gxn[o["middle"] == 0] == 0), "mask disagrees"
    _check_sum(gxn, o["grad_input"], abs_in, O * k * k, "conv grad_input")
    differ = gxn != o["grad_input"]
    extra = float(np.abs(o["grad_input"][differ]).sum()) / np.sqrt(x.numel()) * 2.0 ** -7
    assert abs(gsa - o["grad_scale_a"]) <= 1e-5 * o["grad_scale_a_abs"] + extra + 1e-30, (gsa, o["grad_scale_a"])
    P = B * g.shape[2] * g.shape[3]
    if gw.dtype == torch.bfloat16:
        _check_sum(gw.float().numpy(), o["grad_weight"], abs_w, P, "conv grad_weight")
    else:
        bad = np.abs(gw.double().numpy() - o["grad_weight_exact"]) > P * 2.0 ** -23 * abs_w + 1e-30
        assert not bad.any(), f"conv grad_weight f32: {int(bad.sum())} outside the fp32 bound"
    return differ


CONV_BWD = [(2, 8, 9, 9, 16, 3, 1, 1, 1), (3, 5, 11, 10, 24, 3, 2, 1, 1), (2, 16, 12, 12, 32, 3, 2, 2, 2),
            (1, 3, 7, 7, 8, 1, 1, 0, 1), (4, 32, 14, 14, 64, 3, 1, 1, 1), (2, 4, 6, 6, 8, 5, 1, 2, 1),
            (2, 20, 15, 13, 40, 3, 3, 1, 1)]


@pytest.mark.parametrize("B,C,H,W,O,k,s,p,d", CONV_BWD)
@pytest.mark.parametrize("x_dtype", [torch.bfloat16, torch.float32], ids=["x_bf16", "x_f32"])
def test_conv_backward_matches_oracle(B, C, H, W, O, k, s, p, d, x_dtype):
    differ = _conv_run_and_compare(B, C, H, W, O, k, s, p, d, x_dtype, torch.bfloat16, seed=B + C + H + k)
    assert differ.mean() < 0.01


def test_conv_backward_grad_weight_f32():
    _conv_run_and_compare(2, 16, 12, 12, 32, 3, 2, 1, 1, torch.bfloat16, torch.float32, seed=9)


# The input gradient as one implicit GEMM on the tensor cores (O a multiple of
# 64; conv_dgrad.cu): sub-pixel phases of strides 1 to 4 (and phases no tap
# reaches), dilation, 1x1 to 7x7 kernels, several bands of rows and channel
# tiles, wide rows, channel counts that are not a multiple of 16, O in copies
# of several 64-channel slices or one slice per copy ("slices"), and the route
# it replaces ("gather": the tap matrix D, then the gather).
CONV_BWD_IMPLICIT = [(2, 8, 9, 9, 64, 3, 1, 1, 1), (3, 5, 11, 10, 64, 3, 2, 1, 1), (2, 16, 12, 12, 128, 3, 2, 2, 2),
                     (1, 3, 7, 7, 64, 1, 1, 0, 1), (2, 4, 6, 6, 64, 5, 1, 2, 1), (2, 20, 15, 13, 64, 3, 3, 1, 1),
                     (1, 200, 9, 9, 192, 3, 1, 1, 1), (1, 40, 40, 40, 64, 3, 1, 1, 1), (1, 16, 33, 70, 64, 3, 2, 1, 1),
                     (1, 16, 5, 200, 64, 3, 1, 1, 1), (1, 8, 17, 17, 64, 7, 2, 3, 1), (1, 8, 16, 16, 64, 4, 4, 0, 1),
                     (1, 8, 3, 3, 64, 3, 4, 1, 1), (1, 8, 12, 12, 320, 3, 2, 0, 2), (1, 130, 6, 6, 512, 3, 1, 1, 1),
                     (2, 128, 28, 28, 256, 3, 2, 1, 1), (2, 256, 14, 14, 256, 3, 1, 1, 1)]


@pytest.mark.parametrize("route", ["implicit", "slices", "gather"])
@pytest.mark.parametrize("B,C,H,W,O,k,s,p,d", CONV_BWD_IMPLICIT)
def test_conv_backward_input_gradient_routes(B, C, H, W, O, k, s, p, d, route, monkeypatch):
    monkeypatch.setenv("BT_CONV_DGRAD", route)
    ho, wo = oracle.conv2d_out_size(H, k, s, p, d), oracle.conv2d_out_size(W, k, s, p, d)
    # g per pixel, then the gather route's D or the implicit route's codes of x (16 bytes per 32 channels)
    g_bytes = -(-B * ho * wo * O * 2 // 256) * 256
    codes = -(-B * H * W * -(-C // 32) * 16 // 256) * 256
    ws = bt.bt_binary_conv2d_backward_workspace(B, C, H, W, O, k, s, p, d, True, False)
    assert ws == (g_bytes + -(-C * k * k * B * ho * wo * 4 // 256) * 256 if route == "gather" else g_bytes + codes)
    assert bt.bt_conv2d_backward_implicit(B, C, H, W, O, k, s, p, d) == (route != "gather")
    x_dtype = torch.float32 if (B + C + k) % 2 else torch.bfloat16
    differ = _conv_run_and_compare(B, C, H, W, O, k, s, p, d, x_dtype, torch.bfloat16, seed=B * C + H + s)
    assert differ.mean() < 0.01


@pytest.mark.parametrize("O", [8, 64], ids=["gather", "implicit"])
@pytest.mark.parametrize("x_dtype", [torch.bfloat16, torch.float32], ids=["x_bf16", "x_f32"])
def test_conv_backward_mask_at_the_bound(x_dtype, O):
    # every x on or next to +-scale_a in x's dtype (the consecutive values of
    # the type around it, both signs): the kept set, decided from
    # fp32(x / scale_a) rounded to x's dtype, must be the oracle's exactly.
    # All-positive weights and gradients make every kept gradient nonzero.
    sa = float(np.float32(0.7137))
    if x_dtype == torch.bfloat16:
        base = int(torch.tensor([sa]).to(torch.bfloat16).view(torch.int16).item())
        vals = torch.tensor([base + j for j in range(-12, 13)], dtype=torch.int16).view(torch.bfloat16).float()
    else:
        base = int(np.float32(sa).view(np.int32))
        vals = torch.from_numpy(np.array([base + j for j in range(-12, 13)], dtype=np.int32).view(np.float32))
    vals = torch.cat([vals, -vals])
    B, C, H, W = 1, 4, 5, 5
    x = vals.repeat((B * C * H * W + vals.numel() - 1) // vals.numel())[: B * C * H * W].view(B, C, H, W).to(x_dtype)
    w = torch.ones(O, C, 3, 3, dtype=torch.bfloat16)
    g = torch.ones(B, O, H, W, dtype=torch.bfloat16)
    wst = bt.bt_sign_transpose(w.view(O, -1).to(DEV))
    gx, _, _ = bt.bt_binary_conv2d_backward(x.to(DEV), wst, g.to(DEV), O, 3, 1, 1, 1, sa, 1.0, grad_weight_dtype=None)
    o = oracle.conv2d_backward(x.float().numpy(), w.float().numpy(), g.float().numpy(), sa, 1.0, 1, 1, 1,
                               "bf16" if x_dtype == torch.bfloat16 else "f32")
    kept = gx.cpu().float().numpy() != 0
    assert 0 < int(o["middle"].sum()) < o["middle"].size
    np.testing.assert_array_equal(kept, o["middle"] != 0)


def test_conv_backward_partial_and_empty():
    x, w, g, sa, sw = _conv_inputs(2, 8, 9, 9, 16, 3, 1, 1, 1, torch.bfloat16, 4)
    wst = bt.bt_sign_transpose(w.view(16, -1).to(DEV))
    gx, gsa, gw = bt.bt_binary_conv2d_backward(x.to(DEV), wst, g.to(DEV), 16, 3, 1, 1, 1, sa, sw)
    gx1, _, gw1 = bt.bt_binary_conv2d_backward(x.to(DEV), wst, g.to(DEV), 16, 3, 1, 1, 1, sa, sw, grad_weight_dtype=None)
    _, _, gw2 = bt.bt_binary_conv2d_backward(x.to(DEV), None, g.to(DEV), 16, 3, 1, 1, 1, sa, sw, grad_input=False)
    assert gw1 is None and torch.equal(gx1.cpu(), gx.cpu()) and torch.equal(gw2.cpu(), gw.cpu())
    e = torch.empty(0, 8, 9, 9, dtype=torch.bfloat16, device=DEV)
    ge = torch.empty(0, 16, 9, 9, dtype=torch.bfloat16, device=DEV)
    gxe, gsae, gwe = bt.bt_binary_conv2d_backward(e, wst, ge, 16, 3, 1, 1, 1, sa, sw)
    assert gxe.numel() == 0 and float(gsae.cpu()) == 0.0 and torch.all(gwe.cpu() == 0)


@pytest.mark.slow
def test_conv_backward_full_size_sampled():
    # the stride-2 layer at full size as the benchmark runs it (its x and W,
    # an N(0, 0.01) bf16 upstream gradient): grad_input of four whole images
    # (each depends on its own g alone), sampled grad_weight entries, and
    # grad_scale_a recomputed from the GPU's own grad_input
    wl = workloads.NAMED["downsample_conv"]()
    x, w = wl.x, wl.w
    B, C, H, W = x.shape
    O, _, k, _ = w.shape
    s, p, d = wl.stride, wl.padding, wl.dilation
    ho, wo = oracle.conv2d_out_size(H, k, s, p, d), oracle.conv2d_out_size(W, k, s, p, d)
    gen = torch.Generator().manual_seed(31)
    g = (torch.randn(B, O, ho, wo, generator=gen) * 0.01).to(torch.bfloat16)
    sa, sw = wl.scale_a, wl.scale_w
    wst = bt.bt_sign_transpose(w.reshape(O, -1).to(DEV))
    gx, gsa, gw = bt.bt_binary_conv2d_backward(x.to(DEV), wst, g.to(DEV), O, k, s, p, d, sa, sw)
    torch.cuda.synchronize()
    gx, gsa, gw = gx.cpu(), float(gsa.cpu()), gw.cpu()
    imgs = np.array([0, 1, 127, B - 1])
    o = oracle.conv2d_backward(x[imgs].float().numpy(), w.float().numpy(), g[imgs].float().numpy(), sa, sw, s, p, d,
                               "bf16")
    bw = float(oracle.bf16_round(np.float32(sw)))
    abs_in = torch.nn.grad.conv2d_input((len(imgs), C, H, W), torch.full(w.shape, bw, dtype=torch.float64),
                                        g[imgs].double().abs(), stride=s, padding=p, dilation=d).numpy()
    gxs = gx[imgs].float().numpy()
    assert np.all(gxs[o["middle"] == 0] == 0), "mask disagrees"
    _check_sum(gxs, o["grad_input"], abs_in, O * k * k, "conv grad_input images")
    rng = np.random.default_rng(5)
    oi = np.concatenate([rng.integers(0, O, 600), [0, 0, O - 1, O - 1]])
    ti = np.concatenate([rng.integers(0, C * k * k, 600), [0, C * k * k - 1, 0, C * k * k - 1]])
    want = oracle.conv2d_grad_weight_at(x.float().numpy(), g.float().numpy(), sa, s, p, d, k, oi, ti)
    ba = float(oracle.bf16_round(np.float32(sa)))
    bound = g.double().abs().sum(dim=(0, 2, 3)).numpy()[oi] * ba
    _check_sum(gw.reshape(O, -1).float().numpy()[oi, ti], oracle.bf16_round(want), bound, B * ho * wo,
               "conv grad_weight entries")
    xf = x.float().numpy()
    terms = ((gx.float().numpy() * oracle.sign(xf)).astype(np.float32) * np.float32(1.0 / np.sqrt(x.numel())))
    terms = terms.astype(np.float64)
    assert abs(gsa - terms.sum()) <= 1e-5 * np.abs(terms).sum()


@pytest.mark.slow
def test_conv_backward_stride2_layer_slice():
    # 16 images of the stride-2 downsampling layer [256,128,28,28] x [256,128,3,3]
    _conv_run_and_compare(16, 128, 28, 28, 256, 3, 2, 1, 1, torch.bfloat16, torch.bfloat16, seed=21)
