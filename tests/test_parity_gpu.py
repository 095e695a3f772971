"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Integer results (packed operands, raw dot products) must match bit for bit;
scaled float outputs within 1e-6 relative (the epilogue is one fp32 multiply
and one round-to-nearest-even cast on both sides, so they match exactly in
practice). Sizes span several 128 x 128 tiles with ragged tails; the full
workloads are checked at every output against the oracle's whole forward.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

import xnor_popcount_gemm_gb300 as bt

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
REL_TOL = 1e-6
OUT_T = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16, "i32": torch.int32}
CODES = [bt.BT_CODE_BITS, bt.BT_CODE_E4M3, bt.BT_CODE_E2M1]
CODE_IDS = ["bits", "e4m3", "e2m1"]
TC_CODES = [bt.BT_CODE_E4M3, bt.BT_CODE_E2M1]


@pytest.fixture(autouse=True)
def _device_clean():
    yield
    assert bt.bt_device_status() == 0


def assert_close_rel(got: torch.Tensor, want: torch.Tensor):
    assert got.shape == want.shape and got.dtype == want.dtype
    if got.dtype == torch.int32:
        assert torch.equal(got, want)
        return
    g, w = got.double(), want.double()
    err = (g - w).abs()
    bad = err > REL_TOL * w.abs()
    assert not bad.any(), f"{int(bad.sum())} mismatches, first at {bad.nonzero()[0].tolist()}"


def _gen(seed, shape, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(dtype)


# ---------------------------------------------------------------------------
# Packing
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("K", [1, 7, 31, 32, 33, 100, 255, 256, 257, 1000, 4100])
def test_pack_rows(code, dtype, K):
    x = _gen(K, (37, K), dtype)
    x[0, : min(K, 6)] = torch.tensor([0.0, -0.0, float("nan"), float("inf"), -float("inf"), -1e-30])[: min(K, 6)].to(dtype)
    for bias in (None, torch.tensor([0.05]), torch.linspace(-0.2, 0.2, K)):
        got = bt.bt_pack_sign(x.to(DEV), code, bt.BT_LAYOUT_ROWS,
                              None if bias is None else bias.to(DEV)).cpu().numpy()
        want = oracle.pack_rows(oracle.binarize(x, bias, channel_axis=-1), code)
        np.testing.assert_array_equal(got, want)


# Shifts around which the sign decision is delicate: values of -b that the
# input type cannot represent (the comparison must round them the right way),
# ones it can (x = -b gives +1), signed zeros, a subnormal, values past the
# fp16 range, the fp32 extremes, and non-finite shifts.
EDGE_SHIFTS = [0.05, -0.1, 0.125, -0.0, 0.0, 1e-40, -1e-40, 65504.0, 70000.0, -70000.0, 1.0000001,
               3.0e38, -3.0e38, float("inf"), -float("inf"), float("nan")]


def _all_16bit(dtype):
    """Every bit pattern of a 2-byte float type, as a [64, 1024] tensor."""
    bits = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    return bits.view(dtype).reshape(64, 1024)


def _near_f32(values):
    """fp32 values next to each of `values` (4 steps either way) and the specials."""
    out = [0.0, -0.0, float("inf"), -float("inf"), float("nan"), 1e-45, -1e-45, 3.4e38, -3.4e38]
    for v in values:
        t = torch.tensor([v], dtype=torch.float32)
        for direction in (float("inf"), -float("inf")):
            u = t.clone()
            for _ in range(4):
                u = torch.nextafter(u, torch.tensor([direction]))
                out.append(float(u))
        out.append(float(t))
    x = torch.tensor(out, dtype=torch.float32)
    pad = (-x.numel()) % 64
    return torch.cat([x, torch.zeros(pad)]).reshape(-1, 64)


@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_pack_rows_sign_decision_edges(code, dtype):
    # 2-byte inputs: every bit pattern against every edge shift; fp32: the
    # neighbours of -b. Scalar shifts use the threshold comparison (finite) or
    # the fp32 sum (non-finite); both must equal the oracle's sign of x + b.
    for b in EDGE_SHIFTS:
        x = _all_16bit(dtype) if dtype != torch.float32 else _near_f32([-b] + [-v for v in EDGE_SHIFTS])
        bias = torch.tensor([b], dtype=torch.float32)
        got = bt.bt_pack_sign(x.to(DEV), code, bt.BT_LAYOUT_ROWS, bias.to(DEV)).cpu().numpy()
        want = oracle.pack_rows(oracle.binarize(x, bias, channel_axis=-1), code)
        np.testing.assert_array_equal(got, want, err_msg=f"shift {b}")
    # a per-column shift holding all of them at once
    x = _all_16bit(dtype) if dtype != torch.float32 else _near_f32([-v for v in EDGE_SHIFTS])
    cols = torch.tensor(EDGE_SHIFTS, dtype=torch.float32).repeat(x.shape[1] // len(EDGE_SHIFTS) + 1)[: x.shape[1]]
    got = bt.bt_pack_sign(x.to(DEV), code, bt.BT_LAYOUT_ROWS, cols.to(DEV)).cpu().numpy()
    want = oracle.pack_rows(oracle.binarize(x, cols, channel_axis=-1), code)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_pack_nhwc_sign_decision_edges(code, dtype):
    # every bit pattern as NCHW [4, 16, 32, 32], against each edge shift as a
    # scalar and against all of them as the 16 per-channel shifts
    x = _all_16bit(dtype).reshape(4, 16, 32, 32)
    for bias in [torch.tensor([b], dtype=torch.float32) for b in EDGE_SHIFTS] + \
            [torch.tensor(EDGE_SHIFTS, dtype=torch.float32)]:
        got = bt.bt_pack_sign(x.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC, bias.to(DEV)).cpu().numpy()
        want = oracle.pack_nchw_to_nhwc(oracle.binarize(x, bias, channel_axis=1), code)
        np.testing.assert_array_equal(got, want, err_msg=f"shift {bias.tolist()}")


@pytest.mark.parametrize("impl", ["default", "warp", "smem"])
@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("shape", [(2, 3, 5, 5), (3, 37, 4, 4), (2, 64, 14, 14), (1, 130, 7, 9),
                                   (4, 256, 3, 3), (2, 128, 28, 28), (1, 700, 10, 10), (1, 6200, 3, 3),
                                   (2, 33, 2, 2), (3, 96, 8, 12), (2, 96, 40, 40)])
def test_pack_nchw_to_nhwc(code, dtype, shape, impl, monkeypatch):
    # planes whose bytes are a multiple of 16 take a warp-level kernel (32
    # pixels x 32 channels per warp: for E2M1 the one shared with the
    # convolution's packing warps, else, and with BT_PACK_NHWC=warp, the
    # byte-mask one) unless BT_PACK_NHWC=smem; the others take the
    # shared-memory transpose
    if impl == "default":
        monkeypatch.delenv("BT_PACK_NHWC", raising=False)
    else:
        monkeypatch.setenv("BT_PACK_NHWC", impl)
    x = _gen(sum(shape), shape, dtype)
    for bias in (None, torch.tensor([-0.1]), torch.linspace(-0.3, 0.3, shape[1])):
        got = bt.bt_pack_sign(x.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC,
                              None if bias is None else bias.to(DEV)).cpu().numpy()
        want = oracle.pack_nchw_to_nhwc(oracle.binarize(x, bias, channel_axis=1), code)
        np.testing.assert_array_equal(got, want)


def _unfold_expected(x, bias, code, k, s, p, d):
    """The im2col rows of the oracle's packed pixels: row (b, ho, wo), tap
    (kh, kw) holds pixel (ho*s - p + kh*d, wo*s - p + kw*d), zeros in the padding."""
    pix = oracle.pack_nchw_to_nhwc(oracle.binarize(x, bias, channel_axis=1), code)   # [B, H, W, rbc]
    B, H, W, rbc = pix.shape
    Ho, Wo = bt.conv2d_out_size(H, k, s, p, d), bt.conv2d_out_size(W, k, s, p, d)
    rows = np.zeros((B, Ho, Wo, k, k, rbc), dtype=np.uint8)
    for kh in range(k):
        for kw in range(k):
            for ho in range(Ho):
                hi = ho * s - p + kh * d
                if not 0 <= hi < H:
                    continue
                for wo in range(Wo):
                    wi = wo * s - p + kw * d
                    if 0 <= wi < W:
                        rows[:, ho, wo, kh, kw] = pix[:, hi, wi]
    return rows.reshape(B * Ho * Wo, k * k * rbc)


IM2COL_SHAPES = [
    # B, C, H, W, k, s, p, d, dtype
    (2, 128, 28, 28, 3, 2, 1, 1, torch.bfloat16), (2, 128, 28, 28, 3, 2, 2, 2, torch.bfloat16),
    (2, 256, 14, 14, 3, 1, 1, 1, torch.float32), (3, 64, 14, 14, 3, 1, 1, 1, torch.float16),
    (2, 70, 13, 13, 3, 2, 1, 2, torch.bfloat16), (1, 33, 9, 7, 5, 3, 3, 1, torch.float32),
    (2, 31, 8, 8, 1, 1, 0, 1, torch.bfloat16), (1, 40, 12, 10, 3, 2, 0, 1, torch.float32),
    (2, 3, 5, 5, 3, 1, 1, 1, torch.bfloat16),       # planes not 16-byte aligned: direct kernel
    (1, 700, 10, 10, 3, 1, 1, 1, torch.float32),    # band too wide for shared memory: direct kernel
    (1, 16, 4, 4, 1, 1, 3, 1, torch.bfloat16),      # taps far into the padding
]


@pytest.mark.parametrize("code", TC_CODES, ids=["e4m3", "e2m1"])
@pytest.mark.parametrize("B,C,H,W,k,s,p,d,dtype", IM2COL_SHAPES)
def test_pack_im2col(code, B, C, H, W, k, s, p, d, dtype):
    x = _gen(B + C + H + k, (B, C, H, W), dtype)
    x[0, 0, 0, : min(W, 3)] = torch.tensor([0.0, -0.0, float("nan")])[: min(W, 3)].to(dtype)
    for bias in (None, torch.tensor([0.05]), torch.linspace(-0.2, 0.2, C)):
        got = bt.bt_pack_im2col(x.to(DEV), code, k, s, p, d, None if bias is None else bias.to(DEV)).cpu().numpy()
        np.testing.assert_array_equal(got, _unfold_expected(x, bias, code, k, s, p, d))


@pytest.mark.parametrize("code", TC_CODES, ids=["e4m3", "e2m1"])
def test_conv_from_im2col_rows(code):
    B, C, H, W, O, k, s, p, d = 3, 96, 15, 15, 70, 3, 2, 1, 1
    x = _gen(21, (B, C, H, W), torch.bfloat16)
    w = _gen(22, (O, C, k, k), torch.bfloat16)
    rows = bt.bt_pack_im2col(x.to(DEV), code, k, s, p, d)
    wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    assert bt.bt_binary_conv2d_workspace(B, C, H, W, k, s, p, d, bt.BT_PACKED_IM2COL, code) == 0
    got = bt.bt_binary_conv2d(rows, wp, code, C, k, s, p, d, 1.0, 1.0, out_dtype=torch.int32,
                              x_im2col_hw=(B, H, W)).cpu()
    want = oracle.conv2d_dot(oracle.binarize(x), oracle.binarize_weight(w), s, p, d)
    assert torch.equal(got, torch.from_numpy(want))


# ---------------------------------------------------------------------------
# Linear
# ---------------------------------------------------------------------------

def gpu_linear(x, w, code, scale_a, scale_w, bias, out_dtype, algo=bt.BT_ALGO_AUTO):
    wp = bt.bt_pack_sign(w.to(DEV), code)
    y = bt.bt_binary_linear(x.to(DEV), wp, code, x.shape[1], scale_a, scale_w,
                            None if bias is None else bias.to(DEV), out_dtype=OUT_T[out_dtype],
                            algo=algo)
    return y.cpu()


LIN_SHAPES = [(1, 1, 1), (5, 7, 33), (130, 129, 257), (256, 384, 4100), (300, 200, 1000),
              (129, 257, 96), (64, 256, 512), (17, 600, 2049)]


@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
@pytest.mark.parametrize("M,N,K", LIN_SHAPES)
def test_linear_matches_oracle(code, M, N, K):
    x = _gen(M + N + K, (M, K), torch.bfloat16)
    w = _gen(M * N + K, (N, K), torch.bfloat16) * 0.02
    bias = torch.tensor([0.03])
    sa, sw = workloads.mean_abs(x), workloads.mean_abs(w)
    for od in ("i32", "f32", "bf16", "f16"):
        got = gpu_linear(x, w, code, sa, sw, bias, od)
        want = oracle.binary_linear(x, w, sa, sw, bias, od)
        assert_close_rel(got, want)


@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
def test_linear_f32_input_per_column_bias(code):
    M, N, K = 150, 140, 333
    x = _gen(1, (M, K))
    w = _gen(2, (N, K))
    bias = torch.linspace(-0.5, 0.5, K)
    got = gpu_linear(x, w, code, 0.75, 1.25, bias, "f32")
    assert_close_rel(got, oracle.binary_linear(x, w, 0.75, 1.25, bias, "f32"))


@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
@pytest.mark.parametrize("K", [4096, 11008, 16384])
def test_linear_extreme_sums_are_exact(code, K):
    # rows equal to (or the negation of) weight rows drive every partial sum to
    # its largest magnitude; dot must still be exactly +-K.
    if code != bt.BT_CODE_BITS and K > 16384:
        pytest.skip("beyond the tensor-core bound")
    w = _gen(K, (128, K))
    x = torch.cat([w[:64], -w[64:]])
    x = torch.where(x == 0, torch.ones_like(x), x)
    w = torch.where(w == 0, torch.ones_like(w), w)
    got = gpu_linear(x, w, code, 1.0, 1.0, None, "i32")
    want = oracle.linear_dot(oracle.binarize(x), oracle.binarize_weight(w))
    assert torch.equal(got, torch.from_numpy(want))
    d = got.diagonal()
    assert (d[:64] == K).all() and (d[64:] == -K).all()


@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
def test_linear_prepacked_input(code):
    M, N, K = 200, 136, 700
    x, w = _gen(3, (M, K)), _gen(4, (N, K))
    xp = bt.bt_pack_sign(x.to(DEV), code)
    wp = bt.bt_pack_sign(w.to(DEV), code)
    y = bt.bt_binary_linear(xp, wp, code, K, 1.0, 1.0, out_dtype=torch.int32, x_packed=True).cpu()
    want = oracle.linear_dot(oracle.binarize(x), oracle.binarize_weight(w))
    assert torch.equal(y, torch.from_numpy(want))


def test_linear_empty_and_errors():
    w = bt.bt_pack_sign(torch.randn(8, 64, device=DEV), bt.BT_CODE_BITS)
    y = bt.bt_binary_linear(torch.randn(0, 64, device=DEV), w, bt.BT_CODE_BITS, 64, 1.0, 1.0)
    assert y.shape == (0, 8)
    with pytest.raises(bt.BtError):
        bt.bt_binary_linear(torch.randn(4, 64, device=DEV), w, bt.BT_CODE_BITS, 64, 0.0, 1.0)
    with pytest.raises(bt.BtError):
        bt.bt_binary_linear(torch.randn(4, 64, device=DEV), w, bt.BT_CODE_BITS, 64, 1.0, 1.0,
                            algo=bt.BT_ALGO_TC_E2M1)


# ---------------------------------------------------------------------------
# Conv
# ---------------------------------------------------------------------------

def gpu_conv(x, w, code, s, p, d, scale_a, scale_w, bias, out_dtype):
    wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    y = bt.bt_binary_conv2d(x.to(DEV), wp, code, x.shape[1], w.shape[2], s, p, d, scale_a, scale_w,
                            None if bias is None else bias.to(DEV), out_dtype=OUT_T[out_dtype])
    return y.cpu()


CONV_SHAPES = [
    # B, C, H, W, O, k, s, p, d
    (2, 3, 5, 5, 4, 3, 1, 1, 1), (2, 70, 13, 13, 130, 3, 2, 1, 2), (1, 33, 9, 7, 5, 5, 3, 3, 1),
    (3, 64, 14, 14, 129, 3, 1, 1, 1), (1, 256, 6, 6, 64, 3, 1, 1, 1), (2, 128, 11, 11, 40, 3, 2, 2, 2),
    (1, 5, 1, 1, 3, 3, 1, 1, 1), (2, 31, 8, 8, 7, 1, 1, 0, 1), (1, 40, 12, 10, 33, 3, 2, 0, 1),
]


@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
@pytest.mark.parametrize("B,C,H,W,O,k,s,p,d", CONV_SHAPES)
def test_conv_matches_oracle(code, B, C, H, W, O, k, s, p, d):
    x = _gen(B + C + H, (B, C, H, W), torch.bfloat16)
    w = _gen(O + k, (O, C, k, k), torch.bfloat16)
    bias = torch.linspace(-0.1, 0.1, C)
    sa, sw = workloads.mean_abs(x), workloads.mean_abs(w)
    for od in ("i32", "f32", "bf16"):
        got = gpu_conv(x, w, code, s, p, d, sa, sw, bias, od)
        want = oracle.binary_conv2d(x, w, sa, sw, s, p, d, bias, od)
        assert_close_rel(got, want)


@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
def test_conv_f32_scalar_bias(code):
    x, w = _gen(5, (2, 48, 10, 10)), _gen(6, (24, 48, 3, 3))
    bias = torch.tensor([0.2])
    got = gpu_conv(x, w, code, 1, 1, 1, 0.5, 2.0, bias, "f32")
    assert_close_rel(got, oracle.binary_conv2d(x, w, 0.5, 2.0, 1, 1, 1, bias, "f32"))


@pytest.mark.parametrize("implicit", ["1", "0"])
@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
def test_conv_prepacked_input(code, implicit, monkeypatch):
    # packed NHWC pixels in, through a caller workspace sized by the query:
    # none for the popcount path and the implicit-im2col contraction, the
    # im2col rows for the explicit unfold (BT_CONV_IMPLICIT=0)
    monkeypatch.setenv("BT_CONV_IMPLICIT", implicit)
    B, C, H, W, O, k, s, p, d = 2, 96, 9, 11, 50, 3, 2, 1, 1
    x = _gen(11, (B, C, H, W), torch.bfloat16)
    w = _gen(12, (O, C, k, k), torch.bfloat16)
    xp = bt.bt_pack_sign(x.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    wp = bt.bt_pack_sign(w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    nbytes = bt.bt_binary_conv2d_workspace(B, C, H, W, k, s, p, d, bt.BT_PACKED, code)
    assert (nbytes == 0) == (code == bt.BT_CODE_BITS or implicit == "1")
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=DEV) if nbytes else None
    got = bt.bt_binary_conv2d(xp, wp, code, C, k, s, p, d, 1.0, 1.0, out_dtype=torch.int32, x_packed=True,
                              workspace=ws).cpu()
    want = oracle.conv2d_dot(oracle.binarize(x), oracle.binarize_weight(w), s, p, d)
    assert torch.equal(got, torch.from_numpy(want))


# ---------------------------------------------------------------------------
# Full-size workloads, in the launch configuration the benchmark times: every
# integer output bit for bit and every scaled output against the oracle's
# whole forward (computed once per workload and shared by the codes).
# ---------------------------------------------------------------------------

_ORACLE_DOT = {}


def _oracle_dot(name):
    if name not in _ORACLE_DOT:
        _ORACLE_DOT.clear()                 # one full-size result held at a time
        wl = workloads.NAMED[name]()
        if wl.kind == "linear":
            sa = oracle.binarize(wl.x, wl.bias, channel_axis=-1)
            _ORACLE_DOT[name] = oracle.linear_dot(sa, oracle.binarize_weight(wl.w))
        else:
            sa = oracle.binarize(wl.x, wl.bias, channel_axis=1)
            _ORACLE_DOT[name] = oracle.conv2d_dot(sa, oracle.binarize_weight(wl.w), wl.stride, wl.padding,
                                                  wl.dilation)
    return _ORACLE_DOT[name]


@pytest.mark.slow
@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
@pytest.mark.parametrize("name", ["llm_linear", "large_linear", "ragged_linear", "tiny_linear"])
def test_full_linear_workloads(name, code):
    wl = workloads.NAMED[name]()
    M, N, K = wl.gemm_shape()
    wp = bt.bt_pack_sign(wl.w.to(DEV), code)
    xd = wl.x.to(DEV)
    bias = None if wl.bias is None else wl.bias.to(DEV)
    dot = bt.bt_binary_linear(xd, wp, code, K, wl.scale_a, wl.scale_w, bias, out_dtype=torch.int32).cpu()
    y = bt.bt_binary_linear(xd, wp, code, K, wl.scale_a, wl.scale_w, bias,
                            out_dtype=OUT_T[wl.out_dtype]).cpu()
    want = _oracle_dot(name)
    np.testing.assert_array_equal(dot.numpy(), want)
    assert_close_rel(y, oracle.epilogue(want, wl.scale_a, wl.scale_w, wl.out_dtype))


@pytest.mark.slow
@pytest.mark.parametrize("fused", ["1", "0"], ids=["fused", "two_kernels"])
@pytest.mark.parametrize("code", CODES, ids=CODE_IDS)
@pytest.mark.parametrize("name", ["resnet_conv", "downsample_conv", "downsample_conv_d2"])
def test_full_conv_workloads(name, code, fused, monkeypatch):
    # float x: one kernel that packs x itself, or (BT_CONV_FUSED=0) the NHWC
    # pack kernel, then the contraction of the packed pixels
    if code == bt.BT_CODE_BITS and fused == "0":
        pytest.skip("the popcount route has one form")
    monkeypatch.setenv("BT_CONV_FUSED", fused)
    wl = workloads.NAMED[name]()
    B, C, H, W = wl.x.shape
    O, _, k, _ = wl.w.shape
    wp = bt.bt_pack_sign(wl.w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    xd = wl.x.to(DEV)
    args = (code, C, k, wl.stride, wl.padding, wl.dilation, wl.scale_a, wl.scale_w, None)
    dot = bt.bt_binary_conv2d(xd, wp, *args, out_dtype=torch.int32).cpu()
    y = bt.bt_binary_conv2d(xd, wp, *args, out_dtype=OUT_T[wl.out_dtype]).cpu()
    want = _oracle_dot(name)
    np.testing.assert_array_equal(dot.numpy(), want)
    assert_close_rel(y, oracle.epilogue(want, wl.scale_a, wl.scale_w, wl.out_dtype))


@pytest.mark.slow
@pytest.mark.parametrize("code", TC_CODES, ids=["e4m3", "e2m1"])
@pytest.mark.parametrize("name", ["resnet_conv", "downsample_conv", "downsample_conv_d2"])
def test_full_conv_workloads_bench_calls(name, code):
    """The public calls the benchmark times (one call on x where the
    convolution packs x itself; else the pack, then the contraction of the
    packed activations), every output against the oracle."""
    wl = workloads.NAMED[name]()
    B, C, H, W = wl.x.shape
    O, _, k, _ = wl.w.shape
    wp = bt.bt_pack_sign(wl.w.to(DEV), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
    xd = wl.x.to(DEV)
    geom = (B, C, H, W, k, wl.stride, wl.padding, wl.dilation)
    xt = {torch.float32: bt.BT_F32, torch.bfloat16: bt.BT_BF16}[wl.x.dtype]
    args = (code, C, k, wl.stride, wl.padding, wl.dilation, wl.scale_a, wl.scale_w)
    mode = bt.bt_conv2d_single_pass(*geom, xt, code)
    if mode == 2:
        y = bt.bt_binary_conv2d(xd, wp, *args, out_dtype=OUT_T[wl.out_dtype])
    elif mode == 1:
        rows = bt.bt_pack_im2col(xd, code, k, wl.stride, wl.padding, wl.dilation)
        y = bt.bt_binary_conv2d(rows, wp, *args, out_dtype=OUT_T[wl.out_dtype], x_im2col_hw=(B, H, W))
    else:
        xp = bt.bt_pack_sign(xd, code, bt.BT_LAYOUT_NCHW_TO_NHWC)
        y = bt.bt_binary_conv2d(xp, wp, *args, out_dtype=OUT_T[wl.out_dtype], x_packed=True)
    want = _oracle_dot(name)
    assert_close_rel(y.cpu(), oracle.epilogue(want, wl.scale_a, wl.scale_w, wl.out_dtype))


# ---------------------------------------------------------------------------
# Every tile configuration of the tensor-core kernel (the planner picks one
# per shape; BT_TC_CONFIG="bn,d" or "pair,bn,d" forces it): BN columns per
# tile, d 128-byte K slices per pipeline stage; "pair" runs 256-row tiles on
# CTA pairs (cta_group::2). The shapes cover a whole number of slices, a half
# last slice, and rows shorter than one slice.
# ---------------------------------------------------------------------------

TC_CONFIGS = ["240,1", "224,2", "128,4", "64,2", "32,1", "208,2", "96,4", "224,3",
              "pair,240,2", "pair,224,1", "pair,160,4", "pair,128,2", "pair,64,4", "pair,32,1", "pair,208,2",
              "pair,224,3", "pair,240,3", "pair,192,2", "pair,112,2", "pair,96,2", "192,2"]


@pytest.mark.parametrize("epi", ["4", "8"], ids=["epi4", "epi8"])
@pytest.mark.parametrize("cfg", TC_CONFIGS)
@pytest.mark.parametrize("code", TC_CODES, ids=["e4m3", "e2m1"])
def test_linear_tc_configs(cfg, code, epi, monkeypatch):
    # epi: epilogue warps, one or two per TMEM lane quarter (BT_TC_EPI forces
    # either; the planner takes one for aligned rows and long K), on aligned
    # (N = 600, 200, 520) and ragged (N = 330) rows
    monkeypatch.setenv("BT_TC_CONFIG", cfg)
    monkeypatch.setenv("BT_TC_EPI", epi)
    for (M, N, K) in ((700, 600, 1000), (1100, 330, 4100), (300, 200, 100), (260, 520, 700)):
        x = _gen(M + K, (M, K), torch.bfloat16)
        w = _gen(N + K, (N, K), torch.bfloat16)
        sa, sw = workloads.mean_abs(x), workloads.mean_abs(w)
        want_dot = oracle.linear_dot(oracle.binarize(x), oracle.binarize_weight(w))
        got = gpu_linear(x, w, code, sa, sw, None, "i32")
        assert torch.equal(got, torch.from_numpy(want_dot)), (cfg, M, N, K)
        got = gpu_linear(x, w, code, sa, sw, None, "bf16")
        assert_close_rel(got, oracle.epilogue(want_dot, sa, sw, "bf16"))


@pytest.mark.parametrize("cfg", TC_CONFIGS)
@pytest.mark.parametrize("code", TC_CODES, ids=["e4m3", "e2m1"])
def test_conv_tc_configs(cfg, code, monkeypatch):
    monkeypatch.setenv("BT_TC_CONFIG", cfg)
    for (B, C, H, W, O, k, s, p, d) in ((3, 128, 14, 14, 200, 3, 1, 1, 1), (4, 64, 15, 13, 70, 3, 2, 2, 2)):
        x = _gen(B + C, (B, C, H, W), torch.bfloat16)
        w = _gen(O + C, (O, C, k, k), torch.bfloat16)
        want = oracle.conv2d_dot(oracle.binarize(x), oracle.binarize_weight(w), s, p, d)
        got = gpu_conv(x, w, code, s, p, d, 1.0, 1.0, None, "i32")
        assert torch.equal(got, torch.from_numpy(want)), (cfg, B, C, H, W, O)
