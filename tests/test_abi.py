"""CPU checks of the C ABI: the library builds and loads, exports every
function include/bt.h declares, and validates arguments on the host before
it launches anything (no compute call is made here)."""
import ctypes
import os
import re

import pytest
import torch


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
import xnor_popcount_gemm_gb300 as bt


def declared_functions():
    text = open(os.path.join(ROOT, "include", "bt.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bt_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol():
    names = declared_functions()
    assert len(names) >= 10
    lib = ctypes.CDLL(bt.lib_path)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(bt.EXPORTED) == names


def test_version_and_status_strings():
    assert bt.bt_version() >= 100
    for st in range(-6, 1):
        s = bt.bt_status_string(st)
        assert s.startswith("BT_")
    assert "unknown" in bt.bt_status_string(42)


@pytest.mark.parametrize("k,code,want", [
    (1, 0, 16), (32, 0, 16), (128, 0, 16), (129, 0, 32), (4096, 0, 512), (4100, 0, 528),
    (1, 1, 64), (64, 1, 64), (65, 1, 128), (4100, 1, 4160),
    (1, 2, 64), (128, 2, 64), (129, 2, 128), (4100, 2, 2112), (11008, 2, 5504), (256, 2, 128),
])
def test_packed_row_bytes(k, code, want):
    assert bt.bt_packed_row_bytes(k, code) == want


def test_packed_row_bytes_rejects_bad_input():
    assert bt.bt_packed_row_bytes(-1, 0) == -1
    assert bt.bt_packed_row_bytes(5, 7) == -1


def test_workspace_queries(monkeypatch):
    assert bt.bt_binary_linear_workspace(4096, 4096, bt.BT_BF16, bt.BT_CODE_BITS) == 4096 * 512
    assert bt.bt_binary_linear_workspace(3, 33, bt.BT_F32, bt.BT_CODE_BITS) == 256
    assert bt.bt_binary_linear_workspace(10, 10, bt.BT_PACKED, bt.BT_CODE_BITS) == 0
    ws = bt.bt_binary_conv2d_workspace
    # BITS: the packed NHWC pixels only
    assert ws(2, 256, 14, 14, 3, 1, 1, 1, bt.BT_F32, bt.BT_CODE_BITS) == 2 * 14 * 14 * 32
    assert ws(1, 1, 1, 1, 1, 1, 0, 1, bt.BT_F32, bt.BT_CODE_BITS) == 256
    assert ws(1, 1, 1, 1, 1, 1, 0, 1, bt.BT_PACKED, bt.BT_CODE_BITS) == 0
    # E2M1 / E4M3 with the implicit-im2col contraction: the packed pixels only,
    # nothing for packed input
    assert ws(2, 256, 14, 14, 3, 1, 1, 1, bt.BT_F32, bt.BT_CODE_E2M1) == 2 * 14 * 14 * 128
    assert ws(2, 256, 14, 14, 3, 1, 1, 1, bt.BT_PACKED, bt.BT_CODE_E2M1) == 0
    assert ws(2, 128, 28, 28, 3, 2, 1, 1, bt.BT_BF16, bt.BT_CODE_E2M1) == 2 * 28 * 28 * 64
    assert ws(1, 3, 5, 5, 3, 1, 0, 1, bt.BT_F32, bt.BT_CODE_E4M3) == 1792
    # rows wider than one tile (Wo = 298 > 240 columns): packed pixels, then
    # the im2col rows [B*Ho*Wo, k*k*row_bytes(C)] of the explicit unfold
    # (each part rounded up to 256 bytes: 298 x 9 x 64 = 171648 -> 171776)
    assert ws(1, 16, 3, 300, 3, 1, 0, 1, bt.BT_BF16, bt.BT_CODE_E2M1) == 3 * 300 * 64 + 171776
    # invalid geometry or arguments
    assert ws(1, 8, 4, 4, 0, 1, 0, 1, bt.BT_F32, bt.BT_CODE_E2M1) == 0
    assert ws(1, 8, 4, 4, 3, 0, 0, 1, bt.BT_F32, bt.BT_CODE_E2M1) == 0
    assert ws(1, 8, 4, 4, 3, 1, 0, 1, bt.BT_F32, 7) == 0
    # the explicit unfold (BT_CONV_IMPLICIT=0): pixels, then the rows
    monkeypatch.setenv("BT_CONV_IMPLICIT", "0")
    assert ws(2, 256, 14, 14, 3, 1, 1, 1, bt.BT_F32, bt.BT_CODE_E2M1) == \
        2 * 14 * 14 * 128 + 2 * 14 * 14 * 9 * 128
    assert ws(2, 256, 14, 14, 3, 1, 1, 1, bt.BT_PACKED, bt.BT_CODE_E2M1) == 2 * 14 * 14 * 9 * 128
    # stride 2, padding 1 on 28 x 28 -> 14 x 14 outputs; 128 channels -> 64-byte pixels
    assert ws(2, 128, 28, 28, 3, 2, 1, 1, bt.BT_BF16, bt.BT_CODE_E2M1) == \
        2 * 28 * 28 * 64 + 2 * 14 * 14 * 9 * 64
    # E4M3: one byte per channel; each part rounded up to 256 bytes
    # (25 pixels x 64 B = 1600 -> 1792; 3 x 3 outputs x 9 taps x 64 B = 5184 -> 5376)
    assert ws(1, 3, 5, 5, 3, 1, 0, 1, bt.BT_F32, bt.BT_CODE_E4M3) == 1792 + 5376


# Host validation. Pointers below are never dereferenced: every call fails
# its checks before anything is enqueued.
L = bt._c_lin
C = bt._c_conv
P = bt._c_pack


def lin(**kw):
    a = dict(x=256, xt=bt.BT_F32, w=512, code=0, M=4, N=4, K=8, sa=1.0, sw=1.0, bias=None, blen=0,
             out=768, ot=bt.BT_F32, algo=0, ws=None, wsb=0, s=None)
    a.update(kw)
    return L(*a.values())


def test_linear_validation():
    assert lin(K=0) == bt.BT_ERR_INVALID_ARG
    assert lin(M=-1) == bt.BT_ERR_INVALID_ARG
    assert lin(sa=0.0) == bt.BT_ERR_INVALID_ARG
    assert lin(sw=float("nan")) == bt.BT_ERR_INVALID_ARG
    assert lin(sa=float("inf")) == bt.BT_ERR_INVALID_ARG
    assert lin(sa=-1.0) == bt.BT_ERR_INVALID_ARG
    assert lin(blen=3) == bt.BT_ERR_INVALID_ARG
    assert lin(blen=1, bias=None) == bt.BT_ERR_INVALID_ARG
    assert lin(code=9) == bt.BT_ERR_INVALID_ARG
    assert lin(ot=bt.BT_PACKED) == bt.BT_ERR_INVALID_ARG
    assert lin(xt=bt.BT_I32) == bt.BT_ERR_INVALID_ARG
    assert lin(algo=bt.BT_ALGO_TC_E2M1) == bt.BT_ERR_UNSUPPORTED   # algo does not match BITS
    assert lin(algo=17) == bt.BT_ERR_INVALID_ARG
    assert lin(x=None) == bt.BT_ERR_INVALID_ARG
    assert lin(x=257) == bt.BT_ERR_ALIGNMENT
    assert lin(out=770) == bt.BT_ERR_ALIGNMENT
    assert lin(ws=None) == bt.BT_ERR_WORKSPACE                      # float x needs a workspace
    assert lin(ws=4096, wsb=8) == bt.BT_ERR_WORKSPACE
    assert lin(ws=4096 + 16, wsb=1 << 20) == bt.BT_ERR_ALIGNMENT
    assert lin(K=(1 << 24) + 1) == bt.BT_ERR_UNSUPPORTED
    assert lin(M=0) == bt.BT_OK                                      # empty: nothing to do
    assert lin(N=0, x=None) == bt.BT_OK


def conv(**kw):
    a = dict(x=256, xt=bt.BT_F32, w=512, code=0, B=1, C=3, H=5, W=5, O=2, k=3, s=1, p=1, d=1,
             sa=1.0, sw=1.0, bias=None, blen=0, out=768, ot=bt.BT_F32, algo=0, ws=None, wsb=0,
             st=None)
    a.update(kw)
    return C(*a.values())


def test_conv_validation(monkeypatch):
    assert conv(k=0) == bt.BT_ERR_INVALID_ARG
    assert conv(s=0) == bt.BT_ERR_INVALID_ARG
    assert conv(p=-1) == bt.BT_ERR_INVALID_ARG
    assert conv(d=0) == bt.BT_ERR_INVALID_ARG
    assert conv(H=2, p=0) == bt.BT_ERR_INVALID_ARG        # window larger than the image
    assert conv(blen=2) == bt.BT_ERR_INVALID_ARG
    assert conv(C=0) == bt.BT_ERR_INVALID_ARG
    assert conv(sa=0.0) == bt.BT_ERR_INVALID_ARG
    assert conv(x=264 + 1) == bt.BT_ERR_ALIGNMENT
    assert conv(ws=None) == bt.BT_ERR_WORKSPACE
    # with the explicit unfold (BT_CONV_IMPLICIT=0) the tensor-core codes need
    # the im2col rows even for packed pixels
    monkeypatch.setenv("BT_CONV_IMPLICIT", "0")
    assert conv(xt=bt.BT_PACKED, code=bt.BT_CODE_E2M1, ws=None) == bt.BT_ERR_WORKSPACE
    assert conv(xt=bt.BT_PACKED, code=bt.BT_CODE_E4M3, ws=4096, wsb=1024) == bt.BT_ERR_WORKSPACE
    assert conv(xt=bt.BT_PACKED, code=bt.BT_CODE_E2M1, ws=4096 + 16, wsb=1 << 20) == bt.BT_ERR_ALIGNMENT
    assert conv(B=0) == bt.BT_OK
    assert conv(O=0, x=None) == bt.BT_OK


def test_pack_im2col_validation():
    f = bt._c_pack_im2col
    s = None
    def call(**kw):
        a = dict(x=256, xt=bt.BT_F32, B=1, C=8, H=5, W=5, k=3, st=1, p=1, d=1, bias=None, blen=0,
                 code=bt.BT_CODE_E2M1, out=512, stream=s)
        a.update(kw)
        return f(*a.values())
    assert call(code=bt.BT_CODE_BITS) == bt.BT_ERR_INVALID_ARG      # codes for the tensor cores only
    assert call(xt=bt.BT_PACKED) == bt.BT_ERR_INVALID_ARG
    assert call(C=0) == bt.BT_ERR_INVALID_ARG
    assert call(k=0) == bt.BT_ERR_INVALID_ARG
    assert call(H=1, p=0) == bt.BT_ERR_INVALID_ARG                  # window larger than the image
    assert call(blen=3) == bt.BT_ERR_INVALID_ARG
    assert call(blen=1) == bt.BT_ERR_INVALID_ARG                    # bias length without a bias
    assert call(C=2000) == bt.BT_ERR_UNSUPPORTED                    # C*k*k > 16384
    assert call(x=None) == bt.BT_ERR_INVALID_ARG
    assert call(x=256 + 8) == bt.BT_ERR_ALIGNMENT
    assert call(out=512 + 4) == bt.BT_ERR_ALIGNMENT
    assert call(B=0, x=None, out=None) == bt.BT_OK


def test_conv_im2col_input_validation():
    # pre-unfolded rows: tensor-core codes only, no workspace needed
    assert conv(xt=bt.BT_PACKED_IM2COL, code=bt.BT_CODE_BITS) == bt.BT_ERR_INVALID_ARG
    assert bt.bt_binary_conv2d_workspace(2, 64, 8, 8, 3, 1, 1, 1, bt.BT_PACKED_IM2COL, bt.BT_CODE_E2M1) == 0


def test_conv2d_single_pass_query(monkeypatch):
    q = bt.bt_conv2d_single_pass
    geom = (2, 64, 16, 16, 3, 1, 1, 1)
    assert q(*geom, bt.BT_F32, bt.BT_CODE_BITS) == 0                # popcount convs contract NHWC pixels
    assert q(*geom, bt.BT_PACKED, bt.BT_CODE_E2M1) == 0             # already packed
    assert q(0, 64, 16, 16, 3, 1, 1, 1, bt.BT_F32, bt.BT_CODE_E2M1) == 0
    assert q(2, 64, 1, 1, 3, 1, 0, 1, bt.BT_F32, bt.BT_CODE_E2M1) == 0   # window larger than the image
    assert q(2, 2000, 16, 16, 3, 1, 1, 1, bt.BT_F32, bt.BT_CODE_E2M1) == 0  # K beyond the tensor-core limit
    # one kernel from x (opt-in) where the implicit plan applies and the
    # channel planes are whole 16-byte units; else the NHWC pack runs first
    assert q(*geom, bt.BT_BF16, bt.BT_CODE_E2M1) == 0
    monkeypatch.setenv("BT_CONV_FUSED", "1")
    for code in (bt.BT_CODE_E2M1, bt.BT_CODE_E4M3):
        assert q(*geom, bt.BT_F32, code) == 2
        assert q(*geom, bt.BT_BF16, code) == 2
        assert q(2, 64, 14, 14, 3, 1, 1, 1, bt.BT_BF16, code) == 0     # 392-byte planes
        assert q(2, 64, 14, 14, 3, 1, 1, 1, bt.BT_F32, code) == 2      # 784-byte planes


def test_pack_validation():
    s = None
    assert P(256, bt.BT_F32, 0, 4, 0, 1, 1, None, 0, 0, 512, s) == bt.BT_ERR_INVALID_ARG   # K = 0
    assert P(256, bt.BT_I32, 0, 4, 8, 1, 1, None, 0, 0, 512, s) == bt.BT_ERR_INVALID_ARG
    assert P(256, bt.BT_F32, 5, 4, 8, 1, 1, None, 0, 0, 512, s) == bt.BT_ERR_INVALID_ARG
    assert P(256, bt.BT_F32, 0, 4, 8, 1, 1, None, 3, 0, 512, s) == bt.BT_ERR_INVALID_ARG
    assert P(256, bt.BT_F32, 0, 4, 8, 1, 1, None, 1, 0, 512, s) == bt.BT_ERR_INVALID_ARG
    assert P(None, bt.BT_F32, 0, 4, 8, 1, 1, None, 0, 0, 512, s) == bt.BT_ERR_INVALID_ARG
    assert P(258, bt.BT_F32, 0, 4, 8, 1, 1, None, 0, 0, 512, s) == bt.BT_ERR_ALIGNMENT
    assert P(256, bt.BT_F32, 1, 4, 8, 0, 1, None, 0, 0, 512, s) == bt.BT_ERR_INVALID_ARG
    assert P(None, bt.BT_F32, 0, 0, 8, 1, 1, None, 0, 0, None, s) == bt.BT_OK             # 0 rows


def test_plan():
    code, algo = bt.bt_plan(bt.BT_OP_LINEAR, 4096, 4096, 4096)
    assert code in (0, 1, 2) and algo == {0: bt.BT_ALGO_POPC, 1: bt.BT_ALGO_TC_E4M3,
                                          2: bt.BT_ALGO_TC_E2M1}[code]
    code, algo = bt.bt_plan(bt.BT_OP_LINEAR, 16, 16, 1 << 20)      # K beyond the tensor-core bound
    assert code == bt.BT_CODE_BITS and algo == bt.BT_ALGO_POPC
    with pytest.raises(bt.BtError):
        bt.bt_plan(bt.BT_OP_LINEAR, 0, 1, 1)


def test_plan_override(monkeypatch):
    monkeypatch.setenv("BT_FORCE_ALGO", "popc")
    assert bt.bt_plan(bt.BT_OP_CONV2D, 4096, 256, 2304) == (bt.BT_CODE_BITS, bt.BT_ALGO_POPC)
    monkeypatch.setenv("BT_FORCE_ALGO", "e4m3")
    assert bt.bt_plan(bt.BT_OP_LINEAR, 64, 64, 64) == (bt.BT_CODE_E4M3, bt.BT_ALGO_TC_E4M3)


def test_tune_abi_validation():
    # host-side checks only: no result struct, reps out of range, bad code or
    # dtype, and a zero-row call (a no-op that times and keeps nothing)
    T = bt._c_tune
    res = bt.TuneResult()
    r = ctypes.byref(res)
    args = (None, bt.BT_F32, None, bt.BT_CODE_E2M1, 0, 8, 8, 1.0, 1.0, None, 0, None, bt.BT_F32, None, 0)
    assert T(*args, 5, None, None) == bt.BT_ERR_INVALID_ARG
    assert T(*args, 0, None, r) == bt.BT_ERR_INVALID_ARG
    assert T(*args, 10001, None, r) == bt.BT_ERR_INVALID_ARG
    bad_code = args[:3] + (7,) + args[4:]
    assert T(*bad_code, 5, None, r) == bt.BT_ERR_INVALID_ARG
    assert T(*args, 5, None, r) == bt.BT_OK
    assert res.candidates == 0 and res.us == 0.0 and res.code == bt.BT_CODE_E2M1
    bt.bt_tune_reset()
    assert bt.bt_plan(bt.BT_OP_LINEAR, 16, 16, 1 << 20) == (bt.BT_CODE_BITS, bt.BT_ALGO_POPC)
    # the convolution's: no result struct, reps out of range, a bad code, zero images
    TC = bt._c_tune_conv
    cres = bt.TuneConvResult()
    cr = ctypes.byref(cres)
    cargs = (None, bt.BT_F32, None, bt.BT_CODE_E2M1, 0, 64, 14, 14, 64, 3, 1, 1, 1, 1.0, 1.0, None, 0, None,
             bt.BT_F32, None, 0)
    assert TC(*cargs, 5, None, None) == bt.BT_ERR_INVALID_ARG
    assert TC(*cargs, 0, None, cr) == bt.BT_ERR_INVALID_ARG
    assert TC(*(cargs[:3] + (7,) + cargs[4:]), 5, None, cr) == bt.BT_ERR_INVALID_ARG
    assert TC(*cargs, 5, None, cr) == bt.BT_OK
    assert cres.candidates == 0 and cres.us == 0.0
    # BT_ALGO_TUNE on the forward entry points: the same host checks as AUTO;
    # the variants that take no measured selection refuse it
    L = bt._c_lin
    lin = (None, bt.BT_F32, None, bt.BT_CODE_E2M1, 0, 8, 8, 1.0, 1.0, None, 0, None, bt.BT_F32)
    assert L(*lin, bt.BT_ALGO_TUNE, None, 0, None) == bt.BT_OK                     # zero rows: a no-op
    assert L(*lin[:7], -1.0, *lin[8:], bt.BT_ALGO_TUNE, None, 0, None) == bt.BT_ERR_INVALID_ARG
    assert L(*lin, 5, None, 0, None) == bt.BT_ERR_INVALID_ARG
    C = bt._c_conv
    conv = (None, bt.BT_F32, None, bt.BT_CODE_E2M1, 0, 64, 14, 14, 64, 3, 1, 1, 1, 1.0, 1.0, None, 0, None,
            bt.BT_F32)
    assert C(*conv, bt.BT_ALGO_TUNE, None, 0, None) == bt.BT_OK                     # zero images: a no-op
    # C far past any limit: refused before any size product is formed
    huge = (None, bt.BT_F32, None, bt.BT_CODE_E2M1, 2, 1 << 62, 14, 14, 64, 3, 1, 1, 1, 1.0, 1.0, None, 0, None,
            bt.BT_F32)
    for algo in (bt.BT_ALGO_AUTO, bt.BT_ALGO_TUNE):
        assert C(*huge, algo, None, 0, None) == bt.BT_ERR_UNSUPPORTED
    assert bt.bt_conv2d_single_pass(2, 1 << 62, 14, 14, 3, 1, 1, 1, bt.BT_F32, bt.BT_CODE_E2M1) == 0
    LD = bt._c_lin_ds
    assert LD(None, bt.BT_F32, None, bt.BT_CODE_E2M1, 0, 8, 8, 256, None, 0, None, bt.BT_F32, bt.BT_ALGO_TUNE,
              None, 0, None) == bt.BT_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_device_status_without_device():
    assert bt._c_status(None) == bt.BT_ERR_CUDA


def test_backward_abi_validation():
    assert bt.bt_backward_weight_ld(4093) == 4096 and bt.bt_backward_weight_ld(64) == 64
    assert bt.bt_backward_weight_ld(0) == 0 and bt.bt_backward_weight_ld(-1) == -1
    assert bt.bt_binary_linear_backward_workspace(100, 16, 24, True) == 16 * 128 * 2 + 24 * 128 * 2
    assert bt.bt_binary_linear_backward_workspace(100, 16, 24, False) == 0
    st = bt._c_sign_t
    assert st(256, bt.BT_I32, 4, 4, 8, 512, None) == bt.BT_ERR_INVALID_ARG       # dtype
    assert st(256, bt.BT_F32, 10, 4, 8, 512, None) == bt.BT_ERR_INVALID_ARG      # ld < R
    assert st(256, bt.BT_F32, 4, 4, 12, 512, None) == bt.BT_ERR_INVALID_ARG      # ld not a multiple of 8
    assert st(None, bt.BT_F32, 0, 4, 8, None, None) == bt.BT_OK                  # empty
    assert st(None, bt.BT_F32, 4, 4, 8, 512, None) == bt.BT_ERR_INVALID_ARG
    assert st(256 + 4, bt.BT_F32, 4, 4, 8, 512, None) == bt.BT_ERR_ALIGNMENT
    bw = bt._c_bwd

    def call(**kw):
        a = dict(x=256, xt=bt.BT_BF16, wst=512, ldw=64, g=768, M=16, N=64, K=64, sa=0.5, sw=0.5, gx=1024,
                 gsa=2048, gw=4096, gwt=bt.BT_BF16, ws=8192, wsb=1 << 20, s=None)
        a.update(kw)
        return bw(*a.values())
    assert call(xt=bt.BT_F16) == bt.BT_ERR_INVALID_ARG
    assert call(gwt=bt.BT_I32) == bt.BT_ERR_INVALID_ARG
    assert call(sa=0.0) == bt.BT_ERR_INVALID_ARG
    assert call(sw=float("inf")) == bt.BT_ERR_INVALID_ARG
    assert call(gx=None) == bt.BT_ERR_INVALID_ARG                                # grad_scale_a without grad_x
    assert call(ldw=56) == bt.BT_ERR_INVALID_ARG                                 # ldw < N
    assert call(wst=None) == bt.BT_ERR_INVALID_ARG
    assert call(N=60, ldw=64) == bt.BT_ERR_UNSUPPORTED                           # N not a multiple of 8
    assert call(K=20) == bt.BT_ERR_UNSUPPORTED


def test_conv_backward_abi_validation():
    ws = bt.bt_binary_conv2d_backward_workspace
    assert ws(2, 8, 6, 6, 16, 3, 1, 1, 1, True, True) > 0
    assert ws(2, 8, 6, 6, 16, 3, 1, 1, 1, False, False) == 0
    assert ws(2, 8, 1, 1, 16, 3, 1, 0, 1, True, True) == 0                       # window larger than the image
    f = bt._c_cbwd

    def call(**kw):
        a = dict(x=256, xt=bt.BT_BF16, wst=512, ldw=64, g=768, B=2, C=8, H=6, W=6, O=16, k=3, st=1, p=1, d=1,
                 sa=0.5, sw=0.5, gx=1024, gsa=2048, gw=4096, gwt=bt.BT_BF16, ws=8192, wsb=1 << 24, s=None)
        a.update(kw)
        return f(*a.values())
    assert call(xt=bt.BT_F16) == bt.BT_ERR_INVALID_ARG
    assert call(gwt=bt.BT_I32) == bt.BT_ERR_INVALID_ARG
    assert call(sa=-1.0) == bt.BT_ERR_INVALID_ARG
    assert call(k=0) == bt.BT_ERR_INVALID_ARG
    assert call(H=1, p=0) == bt.BT_ERR_INVALID_ARG                              # empty output
    assert call(O=12) == bt.BT_ERR_UNSUPPORTED                                  # O not a multiple of 8
    assert call(gx=None) == bt.BT_ERR_INVALID_ARG                               # grad_scale_a without grad_x
    assert call(ldw=8) == bt.BT_ERR_INVALID_ARG                                 # ldw < O


def test_device_scale_abi_validation():
    si = bt._c_scale_init
    assert si(256, bt.BT_I32, 10, 2.0, bt.BT_BF16, 512, None) == bt.BT_ERR_INVALID_ARG
    assert si(256, bt.BT_BF16, 10, 2.0, bt.BT_I32, 512, None) == bt.BT_ERR_INVALID_ARG
    assert si(256, bt.BT_BF16, 0, 2.0, bt.BT_BF16, 512, None) == bt.BT_ERR_INVALID_ARG
    assert si(256, bt.BT_BF16, 10, 0.0, bt.BT_BF16, 512, None) == bt.BT_ERR_INVALID_ARG
    assert si(None, bt.BT_BF16, 10, 2.0, bt.BT_BF16, 512, None) == bt.BT_ERR_INVALID_ARG
    assert si(257, bt.BT_BF16, 10, 2.0, bt.BT_BF16, 512, None) == bt.BT_ERR_ALIGNMENT
    ld = bt._c_lin_ds
    assert ld(256, bt.BT_BF16, 512, bt.BT_CODE_E2M1, 4, 4, 64, None, None, 0, 768, bt.BT_BF16, 0, 1024, 4096,
              None) == bt.BT_ERR_INVALID_ARG                                     # no scales
    cd = bt._c_conv_ds
    assert cd(256, bt.BT_BF16, 512, bt.BT_CODE_E2M1, 1, 8, 4, 4, 8, 3, 1, 1, 1, None, None, 0, 768, bt.BT_BF16,
              0, 1024, 1 << 20, None) == bt.BT_ERR_INVALID_ARG


def test_w8a8_abi_validation():
    assert bt.bt_w8a8_conv2d_workspace(2, 8, 6, 6, 16, 3, 1, 1, 1) > 0
    assert bt.bt_w8a8_conv2d_workspace(2, 8, 1, 1, 16, 3, 1, 0, 1) == 0
    f = bt._c_w8

    def call(**kw):
        a = dict(x=256, xt=bt.BT_F32, w=512, wt=bt.BT_F32, B=2, C=8, H=6, W=6, O=16, k=3, s=1, p=1, d=1, sm=0,
                 out=1024, ot=bt.BT_F32, ws=4096, wsb=1 << 24, st=None)
        a.update(kw)
        return f(*a.values())
    assert call(xt=bt.BT_F16) == bt.BT_ERR_INVALID_ARG
    assert call(ot=bt.BT_I32) == bt.BT_ERR_INVALID_ARG
    assert call(k=0) == bt.BT_ERR_INVALID_ARG
    assert call(H=1, p=0) == bt.BT_ERR_INVALID_ARG
    assert call(k=9, H=20, W=20) == bt.BT_ERR_UNSUPPORTED
    assert call(B=0) == bt.BT_OK
    assert call(x=None) == bt.BT_ERR_INVALID_ARG


def test_wait_timeout_setter_validates():
    assert bt._c_wait(61 * 10**9) == bt.BT_ERR_INVALID_ARG
    assert bt._c_wait(0) == bt.BT_OK          # the default (2 s)


def test_first_forward_validation():
    L = bt._c_lin_dsi
    def lin(**kw):
        a = dict(x=256, xt=bt.BT_BF16, w=512, code=bt.BT_CODE_E2M1, M=4, N=4, K=64, scales=1024, factor=2.0,
                 sdt=bt.BT_BF16, bias=None, blen=0, out=2048, ot=bt.BT_F32, algo=0, ws=4096, wsb=1 << 20, s=None)
        a.update(kw)
        return L(*a.values())
    assert lin(scales=None) == bt.BT_ERR_INVALID_ARG
    assert lin(factor=0.0) == bt.BT_ERR_INVALID_ARG
    assert lin(factor=float("inf")) == bt.BT_ERR_INVALID_ARG
    assert lin(sdt=bt.BT_I32) == bt.BT_ERR_INVALID_ARG
    assert lin(xt=bt.BT_PACKED) == bt.BT_ERR_INVALID_ARG          # x must be floats: the scale comes from it
    assert lin(scales=1024 + 4) == bt.BT_ERR_ALIGNMENT
    assert lin(ws=None) == bt.BT_ERR_WORKSPACE
    assert lin(M=0) == bt.BT_OK
    C = bt._c_conv_dsi
    def conv(**kw):
        a = dict(x=256, xt=bt.BT_BF16, w=512, code=bt.BT_CODE_E2M1, B=1, C=8, H=6, W=6, O=4, k=3, st=1, p=1, d=1,
                 scales=1024, factor=2.0, sdt=bt.BT_BF16, bias=None, blen=0, out=2048, ot=bt.BT_F32, algo=0, ws=4096,
                 wsb=1 << 20, s=None)
        a.update(kw)
        return C(*a.values())
    assert conv(scales=None) == bt.BT_ERR_INVALID_ARG
    assert conv(factor=-1.0) == bt.BT_ERR_INVALID_ARG
    assert conv(k=0) == bt.BT_ERR_INVALID_ARG
    assert conv(ws=None) == bt.BT_ERR_WORKSPACE
    assert conv(B=0) == bt.BT_OK



def test_conv2d_backward_implicit_query(monkeypatch):
    # host-side planning only: which route computes grad_x of a geometry
    q = bt.bt_conv2d_backward_implicit
    assert q(256, 128, 28, 28, 256, 3, 2, 1, 1)          # the stride-2 layer: four sub-pixel phases
    assert q(128, 256, 14, 14, 256, 3, 1, 1, 1)          # the stride-1 layer
    assert q(256, 128, 28, 28, 256, 3, 2, 2, 2)          # one phase with all nine taps, three with none
    assert not q(2, 8, 9, 9, 16, 3, 1, 1, 1)             # O not a multiple of 64: tap matrix + gather
    assert not q(2, 8, 9, 9, 64, 3, 5, 1, 1)             # stride above 4
    assert not q(1, 8, 4, 600, 64, 3, 1, 1, 1)           # rows wider than a staged band
    assert not q(0, 8, 9, 9, 64, 3, 1, 1, 1) and not q(2, 8, 9, 9, 64, 3, 1, 1, 0)
    # the workspace follows the route: g per pixel plus the codes of x, or plus the tap matrix
    ws = bt.bt_binary_conv2d_backward_workspace(2, 8, 9, 9, 64, 3, 1, 1, 1, True, False)
    g_bytes, codes = -(-2 * 81 * 64 * 2 // 256) * 256, -(-2 * 81 * 16 // 256) * 256
    assert ws == g_bytes + codes
    monkeypatch.setenv("BT_CONV_DGRAD", "gather")
    assert not q(256, 128, 28, 28, 256, 3, 2, 1, 1)
    assert bt.bt_binary_conv2d_backward_workspace(2, 8, 9, 9, 64, 3, 1, 1, 1, True, False) == \
        g_bytes + -(-8 * 9 * 2 * 81 * 4 // 256) * 256
