"""Python binding of libbt, the binarized linear / conv2d forward for GB300.

Argument marshalling only: every step of the forward runs in the CUDA
kernels of ``_build/libbt.so`` (built from ``csrc/`` by ``build.py``). The
functions keep the C names of ``include/bt.h`` and take torch CUDA tensors;
torch supplies device memory and the current stream. A non-OK status raises
``BtError``. If the library has not been built, importing this package raises:
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "BtError", "lib_path", "BT_F32", "BT_BF16", "BT_F16", "BT_I32", "BT_PACKED", "BT_PACKED_IM2COL",
    "BT_CODE_BITS", "BT_CODE_E4M3", "BT_CODE_E2M1", "BT_LAYOUT_ROWS", "BT_LAYOUT_NCHW_TO_NHWC",
    "BT_ALGO_AUTO", "BT_ALGO_POPC", "BT_ALGO_TC_E4M3", "BT_ALGO_TC_E2M1", "BT_ALGO_TUNE", "BT_OP_LINEAR",
    "BT_OP_CONV2D", "bt_version", "bt_status_string", "bt_packed_row_bytes", "bt_pack_sign",
    "bt_binary_linear_workspace", "bt_binary_linear", "bt_binary_conv2d_workspace",
    "bt_binary_conv2d", "bt_plan", "bt_device_status", "conv2d_out_size", "bt_binary_linear_noalloc",
    "bt_binary_linear_noalloc_max_bytes", "bt_pack_im2col", "bt_conv2d_single_pass", "bt_tune_linear",
    "bt_tune_reset", "bt_tune_conv2d", "bt_conv2d_plan_info", "bt_set_wait_timeout", "bt_binary_linear_dscale_init",
    "bt_binary_conv2d_dscale_init",
]

BT_OK, BT_ERR_INVALID_ARG, BT_ERR_UNSUPPORTED, BT_ERR_ALIGNMENT = 0, -1, -2, -3
BT_ERR_WORKSPACE, BT_ERR_CUDA, BT_ERR_TIMEOUT = -4, -5, -6
BT_F32, BT_BF16, BT_F16, BT_I32, BT_PACKED, BT_PACKED_IM2COL = 0, 1, 2, 3, 4, 5
BT_CODE_BITS, BT_CODE_E4M3, BT_CODE_E2M1 = 0, 1, 2
BT_LAYOUT_ROWS, BT_LAYOUT_NCHW_TO_NHWC = 0, 1
BT_ALGO_AUTO, BT_ALGO_POPC, BT_ALGO_TC_E4M3, BT_ALGO_TC_E2M1, BT_ALGO_TUNE = 0, 1, 2, 3, 4
BT_OP_LINEAR, BT_OP_CONV2D = 0, 1

_DT = {torch.float32: BT_F32, torch.bfloat16: BT_BF16, torch.float16: BT_F16, torch.int32: BT_I32}
_TORCH = {BT_F32: torch.float32, BT_BF16: torch.bfloat16, BT_F16: torch.float16, BT_I32: torch.int32}

lib_path = _build.LIB
if not os.path.exists(lib_path):
    raise ImportError(f"libbt.so is not built ({lib_path}); run xnor_popcount_gemm_gb300.build.build()")

_lib = ctypes.CDLL(lib_path)
_i64, _p, _f, _i, _sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int, ctypes.c_size_t


def _sig(name, res, args):
    fn = getattr(_lib, name)
    fn.restype = res
    fn.argtypes = args
    return fn


_c_version = _sig("bt_version", _i, [])
_c_status_string = _sig("bt_status_string", ctypes.c_char_p, [_i])
_c_row_bytes = _sig("bt_packed_row_bytes", _i64, [_i64, _i])
_c_pack = _sig("bt_pack_sign", _i, [_p, _i, _i, _i64, _i64, _i64, _i64, _p, _i64, _i, _p, _p])
_c_lin_ws = _sig("bt_binary_linear_workspace", _sz, [_i64, _i64, _i, _i])
_c_lin = _sig("bt_binary_linear", _i, [_p, _i, _p, _i, _i64, _i64, _i64, _f, _f, _p, _i64, _p, _i, _i,
                                       _p, _sz, _p])
_c_conv_ws = _sig("bt_binary_conv2d_workspace", _sz, [_i64, _i64, _i64, _i64, _i, _i, _i, _i, _i, _i])
_c_conv = _sig("bt_binary_conv2d", _i, [_p, _i, _p, _i, _i64, _i64, _i64, _i64, _i64, _i, _i, _i, _i,
                                        _f, _f, _p, _i64, _p, _i, _i, _p, _sz, _p])
_c_lin_noalloc = _sig("bt_binary_linear_noalloc", _i, [_p, _i, _p, _i, _i64, _i64, _i64, _f, _f, _p, _i64,
                                                      _p, _i, _i, _p])
_c_noalloc_max = _sig("bt_binary_linear_noalloc_max_bytes", _sz, [])
_c_pack_im2col = _sig("bt_pack_im2col", _i, [_p, _i, _i64, _i64, _i64, _i64, _i, _i, _i, _i, _p, _i64, _i, _p, _p])
_c_single_pass = _sig("bt_conv2d_single_pass", _i, [_i64, _i64, _i64, _i64, _i, _i, _i, _i, _i, _i])
_c_bwd_ld = _sig("bt_backward_weight_ld", _i64, [_i64])
_c_sign_t = _sig("bt_sign_transpose", _i, [_p, _i, _i64, _i64, _i64, _p, _p])
_c_bwd_ws = _sig("bt_binary_linear_backward_workspace", _sz, [_i64, _i64, _i64, _i])
_c_bwd = _sig("bt_binary_linear_backward", _i, [_p, _i, _p, _i64, _p, _i64, _i64, _i64, _f, _f, _p, _p, _p, _i,
                                                _p, _sz, _p])
_c_cbwd_ws = _sig("bt_binary_conv2d_backward_workspace", _sz, [_i64, _i64, _i64, _i64, _i64, _i, _i, _i, _i, _i, _i])
_c_cbwd_impl = _sig("bt_conv2d_backward_implicit", _i, [_i64, _i64, _i64, _i64, _i64, _i, _i, _i, _i])
_c_cbwd = _sig("bt_binary_conv2d_backward", _i, [_p, _i, _p, _i64, _p, _i64, _i64, _i64, _i64, _i64, _i, _i, _i, _i,
                                                 _f, _f, _p, _p, _p, _i, _p, _sz, _p])
_c_scale_init = _sig("bt_scale_init", _i, [_p, _i, _i64, _f, _i, _p, _p])
_c_lin_ds = _sig("bt_binary_linear_dscale", _i, [_p, _i, _p, _i, _i64, _i64, _i64, _p, _p, _i64, _p, _i, _i,
                                                _p, _sz, _p])
_c_conv_ds = _sig("bt_binary_conv2d_dscale", _i, [_p, _i, _p, _i, _i64, _i64, _i64, _i64, _i64, _i, _i, _i, _i,
                                                 _p, _p, _i64, _p, _i, _i, _p, _sz, _p])
_c_lin_dsi = _sig("bt_binary_linear_dscale_init", _i, [_p, _i, _p, _i, _i64, _i64, _i64, _p, _f, _i, _p, _i64, _p,
                                                      _i, _i, _p, _sz, _p])
_c_conv_dsi = _sig("bt_binary_conv2d_dscale_init", _i, [_p, _i, _p, _i, _i64, _i64, _i64, _i64, _i64, _i, _i, _i,
                                                       _i, _p, _f, _i, _p, _i64, _p, _i, _i, _p, _sz, _p])
_c_w8_ws = _sig("bt_w8a8_conv2d_workspace", _sz, [_i64, _i64, _i64, _i64, _i64, _i, _i, _i, _i])
_c_w8 = _sig("bt_w8a8_conv2d", _i, [_p, _i, _p, _i, _i64, _i64, _i64, _i64, _i64, _i, _i, _i, _i, _i, _p, _i, _p,
                                    _sz, _p])
_c_plan = _sig("bt_plan", _i, [_i, _i64, _i64, _i64, ctypes.POINTER(_i), ctypes.POINTER(_i)])


class TuneResult(ctypes.Structure):
    """bt_tune_result: what bt_tune_linear measured and kept."""
    _fields_ = [("code", _i), ("pair", _i), ("bn", _i), ("slices_per_stage", _i), ("epilogue_warps", _i),
                ("candidates", _i), ("us", _f), ("us_model", _f)]


_c_tune = _sig("bt_tune_linear", _i, [_p, _i, _p, _i, _i64, _i64, _i64, _f, _f, _p, _i64, _p, _i, _p, _sz, _i, _p,
                                      ctypes.POINTER(TuneResult)])
_c_tune_reset = _sig("bt_tune_reset", None, [])


class TuneConvResult(ctypes.Structure):
    """bt_tune_conv_result: what bt_tune_conv2d measured and kept."""
    _fields_ = [("code", _i), ("pair", _i), ("weights_resident", _i), ("pixel_stages", _i), ("fused", _i),
                ("candidates", _i), ("us", _f), ("us_model", _f), ("band_split", _i)]


_c_tune_conv = _sig("bt_tune_conv2d", _i, [_p, _i, _p, _i, _i64, _i64, _i64, _i64, _i64, _i, _i, _i, _i, _f, _f, _p,
                                           _i64, _p, _i, _p, _sz, _i, _p, ctypes.POINTER(TuneConvResult)])
_c_status = _sig("bt_device_status", _i, [_p])
_c_wait = _sig("bt_set_wait_timeout", _i, [ctypes.c_uint64])

#: every symbol include/bt.h declares
EXPORTED = ["bt_version", "bt_status_string", "bt_packed_row_bytes", "bt_pack_sign",
            "bt_binary_linear_workspace", "bt_binary_linear", "bt_binary_conv2d_workspace",
            "bt_binary_conv2d", "bt_plan", "bt_device_status", "bt_binary_linear_noalloc",
            "bt_binary_linear_noalloc_max_bytes", "bt_pack_im2col", "bt_conv2d_single_pass", "bt_tune_linear",
            "bt_tune_reset", "bt_tune_conv2d", "bt_conv2d_plan_info",
            "bt_backward_weight_ld", "bt_sign_transpose", "bt_binary_linear_backward_workspace",
            "bt_binary_linear_backward", "bt_binary_conv2d_backward_workspace", "bt_conv2d_backward_implicit",
            "bt_binary_conv2d_backward",
            "bt_scale_init", "bt_binary_linear_dscale", "bt_binary_conv2d_dscale", "bt_w8a8_conv2d_workspace",
            "bt_w8a8_conv2d", "bt_set_wait_timeout", "bt_binary_linear_dscale_init", "bt_binary_conv2d_dscale_init"]


class BtError(RuntimeError):
    def __init__(self, status: int):
        super().__init__(bt_status_string(status))
        self.status = status


def _check(st: int) -> None:
    if st != BT_OK:
        raise BtError(st)


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def bt_version() -> int:
    return int(_c_version())


def bt_status_string(status: int) -> str:
    return _c_status_string(status).decode()


def bt_packed_row_bytes(k: int, code: int) -> int:
    return int(_c_row_bytes(k, code))


def conv2d_out_size(h: int, k: int, s: int, p: int, d: int) -> int:
    return (h + 2 * p - d * (k - 1) - 1) // s + 1


def _contig(t: torch.Tensor, name: str) -> None:
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def bt_pack_sign(x: torch.Tensor, code: int, layout: int = BT_LAYOUT_ROWS, bias=None,
                 out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Shift + sign + pack. ROWS: x [R, K] -> uint8 [R, row_bytes(K)];
    NCHW_TO_NHWC: x [B, C, H, W] -> uint8 [B, H, W, row_bytes(C)]."""
    _contig(x, "x")
    if layout == BT_LAYOUT_ROWS:
        if x.dim() != 2:
            raise ValueError("ROWS layout wants a 2-D x")
        d = (x.shape[0], x.shape[1], 1, 1)
        shape = (x.shape[0], bt_packed_row_bytes(x.shape[1], code))
    else:
        if x.dim() != 4:
            raise ValueError("NCHW_TO_NHWC layout wants a 4-D x")
        d = tuple(x.shape)
        shape = (x.shape[0], x.shape[2], x.shape[3], bt_packed_row_bytes(x.shape[1], code))
    if out is None:
        out = torch.empty(shape, dtype=torch.uint8, device=x.device)
    blen = 0 if bias is None else bias.numel()
    _check(_c_pack(_ptr(x), _DT[x.dtype], layout, *d, _ptr(bias), blen, code, _ptr(out), _stream(stream)))
    return out


def bt_pack_im2col(x: torch.Tensor, code: int, kernel_size: int, stride: int, padding: int, dilation: int,
                   bias=None, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Shift + sign + pack + unfold of NCHW x [B, C, H, W]: the im2col rows
    uint8 [B*Ho*Wo, k*k*row_bytes(C)] a tensor-core conv contracts."""
    _contig(x, "x")
    if x.dim() != 4:
        raise ValueError("bt_pack_im2col wants a 4-D x")
    B, C, H, W = x.shape
    Ho = conv2d_out_size(H, kernel_size, stride, padding, dilation)
    Wo = conv2d_out_size(W, kernel_size, stride, padding, dilation)
    if out is None:
        out = torch.empty((B * max(Ho, 0) * max(Wo, 0), kernel_size * kernel_size * bt_packed_row_bytes(C, code)),
                          dtype=torch.uint8, device=x.device)
    blen = 0 if bias is None else bias.numel()
    _check(_c_pack_im2col(_ptr(x), _DT[x.dtype], B, C, H, W, kernel_size, stride, padding, dilation, _ptr(bias),
                          blen, code, _ptr(out), _stream(stream)))
    return out


def bt_conv2d_single_pass(B: int, C: int, H: int, W: int, kernel_size: int, stride: int, padding: int,
                          dilation: int, x_dtype: int, code: int) -> int:
    """How bt_binary_conv2d splits its work on float x: 2 one kernel from x,
    1 one-pass im2col rows + contraction, 0 NHWC pack + contraction."""
    return int(_c_single_pass(B, C, H, W, kernel_size, stride, padding, dilation, x_dtype, code))


def bt_backward_weight_ld(N: int) -> int:
    return int(_c_bwd_ld(N))


def bt_sign_transpose(w: torch.Tensor, ld: int | None = None, out: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """torch.sign of w [R, C], transposed to bf16 [C, ld] (zeros past R):
    the weight operand of bt_binary_linear_backward (ld defaults to
    bt_backward_weight_ld(R))."""
    _contig(w, "w")
    if w.dim() != 2:
        raise ValueError("bt_sign_transpose wants a 2-D w")
    R, C = w.shape
    ld = bt_backward_weight_ld(R) if ld is None else ld
    if out is None:
        out = torch.empty((C, ld), dtype=torch.bfloat16, device=w.device)
    _check(_c_sign_t(_ptr(w), _DT[w.dtype], R, C, ld, _ptr(out), _stream(stream)))
    return out


def bt_binary_linear_backward_workspace(M: int, N: int, K: int, want_grad_weight: bool = True) -> int:
    return int(_c_bwd_ws(M, N, K, 1 if want_grad_weight else 0))


def bt_binary_linear_backward(x: torch.Tensor, wst: torch.Tensor | None, g: torch.Tensor, scale_a: float,
                              scale_w: float, grad_input: bool = True, grad_weight_dtype=torch.bfloat16,
                              grad_x: torch.Tensor | None = None, grad_scale_a: torch.Tensor | None = None,
                              grad_w: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                              stream=None):
    """Straight-through backward of the binary linear layer for upstream
    gradient g [M, N] (bf16) and forward input x [M, K] (bf16 or f32):
    returns (grad_x [M, K] bf16, grad_scale_a (device float tensor),
    grad_w [N, K]); grad_x / grad_scale_a are None unless grad_input,
    grad_w is None when grad_weight_dtype is None. wst is
    bt_sign_transpose(W)."""
    _contig(x, "x")
    _contig(g, "g")
    M, K = x.shape
    N = g.shape[1]
    if g.shape[0] != M:
        raise ValueError("g and x disagree on M")
    if grad_input:
        if wst is None:
            raise ValueError("grad_input needs wst = bt_sign_transpose(W)")
        _contig(wst, "wst")
        if grad_x is None:
            grad_x = torch.empty((M, K), dtype=torch.bfloat16, device=x.device)
        if grad_scale_a is None:
            grad_scale_a = torch.empty((), dtype=torch.float32, device=x.device)
    else:
        grad_x = grad_scale_a = None
    if grad_weight_dtype is not None and grad_w is None:
        grad_w = torch.empty((N, K), dtype=grad_weight_dtype, device=x.device)
    elif grad_weight_dtype is None:
        grad_w = None
    ws = _workspace(bt_binary_linear_backward_workspace(M, N, K, grad_w is not None), x.device, workspace)
    ldw = wst.shape[1] if (grad_input and wst is not None) else 0
    _check(_c_bwd(_ptr(x), _DT[x.dtype], _ptr(wst) if grad_input else None, ldw, _ptr(g), M, N, K, scale_a,
                  scale_w, _ptr(grad_x), _ptr(grad_scale_a), _ptr(grad_w),
                  _DT[grad_w.dtype] if grad_w is not None else BT_BF16, _ptr(ws),
                  0 if ws is None else ws.numel(), _stream(stream)))
    return grad_x, grad_scale_a, grad_w


def bt_binary_conv2d_backward_workspace(B: int, C: int, H: int, W: int, O: int, kernel_size: int, stride: int,
                                        padding: int, dilation: int, want_grad_input: bool = True,
                                        want_grad_weight: bool = True) -> int:
    return int(_c_cbwd_ws(B, C, H, W, O, kernel_size, stride, padding, dilation, 1 if want_grad_input else 0,
                          1 if want_grad_weight else 0))


def bt_conv2d_backward_implicit(B: int, C: int, H: int, W: int, O: int, kernel_size: int, stride: int, padding: int,
                                dilation: int) -> bool:
    """Whether bt_binary_conv2d_backward computes grad_x of this geometry as
    one implicit GEMM (else the tap matrix and gather route)."""
    return bool(_c_cbwd_impl(B, C, H, W, O, kernel_size, stride, padding, dilation))


def bt_binary_conv2d_backward(x: torch.Tensor, wst: torch.Tensor | None, g: torch.Tensor, O: int, kernel_size: int,
                              stride: int, padding: int, dilation: int, scale_a: float, scale_w: float,
                              grad_input: bool = True, grad_weight_dtype=torch.bfloat16,
                              grad_x: torch.Tensor | None = None, grad_scale_a: torch.Tensor | None = None,
                              grad_w: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                              stream=None):
    """Straight-through backward of the binary conv2d layer: x [B, C, H, W]
    (bf16 or f32), g [B, O, Ho, Wo] bf16, wst = bt_sign_transpose(w.view(O,
    -1)). Returns (grad_x [B, C, H, W] bf16, grad_scale_a (device float
    tensor), grad_w [O, C, k, k]), as bt_binary_linear_backward does."""
    _contig(x, "x")
    _contig(g, "g")
    B, C, H, W = x.shape
    k = kernel_size
    if grad_input:
        if wst is None:
            raise ValueError("grad_input needs wst = bt_sign_transpose(w.view(O, -1))")
        _contig(wst, "wst")
        if grad_x is None:
            grad_x = torch.empty((B, C, H, W), dtype=torch.bfloat16, device=x.device)
        if grad_scale_a is None:
            grad_scale_a = torch.empty((), dtype=torch.float32, device=x.device)
    else:
        grad_x = grad_scale_a = None
    if grad_weight_dtype is not None and grad_w is None:
        grad_w = torch.empty((O, C, k, k), dtype=grad_weight_dtype, device=x.device)
    elif grad_weight_dtype is None:
        grad_w = None
    ws = _workspace(bt_binary_conv2d_backward_workspace(B, C, H, W, O, k, stride, padding, dilation,
                                                        grad_x is not None, grad_w is not None), x.device, workspace)
    ldw = wst.shape[1] if (grad_input and wst is not None) else 0
    _check(_c_cbwd(_ptr(x), _DT[x.dtype], _ptr(wst) if grad_input else None, ldw, _ptr(g), B, C, H, W, O, k, stride,
                   padding, dilation, scale_a, scale_w, _ptr(grad_x), _ptr(grad_scale_a), _ptr(grad_w),
                   _DT[grad_w.dtype] if grad_w is not None else BT_BF16, _ptr(ws), 0 if ws is None else ws.numel(),
                   _stream(stream)))
    return grad_x, grad_scale_a, grad_w


def bt_binary_linear_workspace(M: int, K: int, x_dtype: int, code: int) -> int:
    return int(_c_lin_ws(M, K, x_dtype, code))


def bt_binary_conv2d_workspace(B: int, C: int, H: int, W: int, kernel_size: int, stride: int,
                               padding: int, dilation: int, x_dtype: int, code: int) -> int:
    return int(_c_conv_ws(B, C, H, W, kernel_size, stride, padding, dilation, x_dtype, code))


def _workspace(nbytes: int, device, ws):
    if nbytes == 0:
        return None
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return ws


def bt_binary_linear(x: torch.Tensor, weight: torch.Tensor, w_code: int, K: int, scale_a: float,
                     scale_w: float, bias_a=None, out_dtype=None, algo: int = BT_ALGO_AUTO,
                     x_packed: bool = False, out: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y = cast(fp32(dot * fp32(scale_a*scale_w))) for x [M, K] (or packed rows)
    and a packed weight [N, row_bytes(K)]. Passing a device float tensor
    {scale_a, scale_w} as scale_a (scale_w ignored) reads the scales on the
    device (bt_binary_linear_dscale)."""
    _contig(x, "x")
    _contig(weight, "weight")
    M, N = x.shape[0], weight.shape[0]
    xt = BT_PACKED if x_packed else _DT[x.dtype]
    if out_dtype is None:
        out_dtype = x.dtype if not x_packed else torch.float32
    ot = _DT[out_dtype]
    if out is None:
        out = torch.empty((M, N), dtype=_TORCH[ot], device=x.device)
    ws = _workspace(bt_binary_linear_workspace(M, K, xt, w_code), x.device, workspace)
    blen = 0 if bias_a is None else bias_a.numel()
    if isinstance(scale_a, torch.Tensor):
        # device scales: scale_a is a device float tensor holding {scale_a, scale_w}
        _contig(scale_a, "scales")
        _check(_c_lin_ds(_ptr(x), xt, _ptr(weight), w_code, M, N, K, _ptr(scale_a), _ptr(bias_a), blen,
                         _ptr(out), ot, algo, _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))
        return out
    _check(_c_lin(_ptr(x), xt, _ptr(weight), w_code, M, N, K, scale_a, scale_w, _ptr(bias_a), blen,
                  _ptr(out), ot, algo, _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))
    return out


def bt_binary_conv2d(x: torch.Tensor, weight: torch.Tensor, w_code: int, C: int, kernel_size: int,
                     stride: int, padding: int, dilation: int, scale_a: float, scale_w: float,
                     bias_a=None, out_dtype=None, algo: int = BT_ALGO_AUTO, x_packed: bool = False,
                     out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                     stream=None, x_im2col_hw: tuple | None = None) -> torch.Tensor:
    """NCHW x [B, C, H, W] (or packed NHWC [B, H, W, row_bytes(C)]) with a
    packed weight [O, k, k, row_bytes(C)] -> NCHW [B, O, Ho, Wo]. With
    x_im2col_hw = (B, H, W), x is the rows bt_pack_im2col wrote for an input
    of that batch and size."""
    _contig(x, "x")
    _contig(weight, "weight")
    if x_im2col_hw is not None:
        B, H, W = x_im2col_hw
        xt = BT_PACKED_IM2COL
    elif x_packed:
        B, H, W = x.shape[0], x.shape[1], x.shape[2]
        xt = BT_PACKED
    else:
        B, C2, H, W = x.shape
        if C2 != C:
            raise ValueError("C does not match x")
        xt = _DT[x.dtype]
    O = weight.shape[0]
    if out_dtype is None:
        out_dtype = x.dtype if xt not in (BT_PACKED, BT_PACKED_IM2COL) else torch.float32
    ot = _DT[out_dtype]
    Ho = conv2d_out_size(H, kernel_size, stride, padding, dilation)
    Wo = conv2d_out_size(W, kernel_size, stride, padding, dilation)
    if out is None:
        out = torch.empty((B, O, max(Ho, 0), max(Wo, 0)), dtype=_TORCH[ot], device=x.device)
    ws = _workspace(bt_binary_conv2d_workspace(B, C, H, W, kernel_size, stride, padding, dilation, xt, w_code),
                    x.device, workspace)
    blen = 0 if bias_a is None else bias_a.numel()
    if isinstance(scale_a, torch.Tensor):
        # device scales: scale_a is a device float tensor holding {scale_a, scale_w}
        _contig(scale_a, "scales")
        _check(_c_conv_ds(_ptr(x), xt, _ptr(weight), w_code, B, C, H, W, O, kernel_size, stride, padding,
                          dilation, _ptr(scale_a), _ptr(bias_a), blen, _ptr(out), ot, algo, _ptr(ws),
                          0 if ws is None else ws.numel(), _stream(stream)))
        return out
    _check(_c_conv(_ptr(x), xt, _ptr(weight), w_code, B, C, H, W, O, kernel_size, stride, padding,
                   dilation, scale_a, scale_w, _ptr(bias_a), blen, _ptr(out), ot, algo, _ptr(ws),
                   0 if ws is None else ws.numel(), _stream(stream)))
    return out


def bt_binary_linear_dscale_init(x: torch.Tensor, weight: torch.Tensor, w_code: int, K: int, scales: torch.Tensor,
                                 factor: float = 2.0, scale_dtype=None, bias_a=None, out_dtype=None,
                                 algo: int = BT_ALGO_AUTO, out: torch.Tensor | None = None,
                                 workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """A layer's first forward: scales[0] = (factor * mean|x|) in x's dtype,
    then scale_dtype (x's dtype by default), computed from the read of x that
    packs it; then the forward with alpha = fp32(scales[0] * scales[1])."""
    _contig(x, "x")
    _contig(weight, "weight")
    _contig(scales, "scales")
    M, N = x.shape[0], weight.shape[0]
    xt = _DT[x.dtype]
    st = _DT[scale_dtype if scale_dtype is not None else x.dtype]
    ot = _DT[out_dtype if out_dtype is not None else x.dtype]
    if out is None:
        out = torch.empty((M, N), dtype=_TORCH[ot], device=x.device)
    ws = _workspace(bt_binary_linear_workspace(M, K, xt, w_code), x.device, workspace)
    blen = 0 if bias_a is None else bias_a.numel()
    _check(_c_lin_dsi(_ptr(x), xt, _ptr(weight), w_code, M, N, K, _ptr(scales), factor, st, _ptr(bias_a), blen,
                      _ptr(out), ot, algo, _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))
    return out


def bt_binary_conv2d_dscale_init(x: torch.Tensor, weight: torch.Tensor, w_code: int, kernel_size: int, stride: int,
                                 padding: int, dilation: int, scales: torch.Tensor, factor: float = 2.0,
                                 scale_dtype=None, bias_a=None, out_dtype=None, algo: int = BT_ALGO_AUTO,
                                 out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                                 stream=None) -> torch.Tensor:
    """The conv2d form of bt_binary_linear_dscale_init (NCHW x, packed weight
    [O, k, k, row_bytes(C)], NCHW out)."""
    _contig(x, "x")
    _contig(weight, "weight")
    _contig(scales, "scales")
    B, C, H, W = x.shape
    O = weight.shape[0]
    xt = _DT[x.dtype]
    st = _DT[scale_dtype if scale_dtype is not None else x.dtype]
    ot = _DT[out_dtype if out_dtype is not None else x.dtype]
    Ho = conv2d_out_size(H, kernel_size, stride, padding, dilation)
    Wo = conv2d_out_size(W, kernel_size, stride, padding, dilation)
    if out is None:
        out = torch.empty((B, O, max(Ho, 0), max(Wo, 0)), dtype=_TORCH[ot], device=x.device)
    ws = _workspace(bt_binary_conv2d_workspace(B, C, H, W, kernel_size, stride, padding, dilation, xt, w_code),
                    x.device, workspace)
    blen = 0 if bias_a is None else bias_a.numel()
    _check(_c_conv_dsi(_ptr(x), xt, _ptr(weight), w_code, B, C, H, W, O, kernel_size, stride, padding, dilation,
                       _ptr(scales), factor, st, _ptr(bias_a), blen, _ptr(out), ot, algo, _ptr(ws),
                       0 if ws is None else ws.numel(), _stream(stream)))
    return out


def bt_w8a8_conv2d_workspace(B: int, C: int, H: int, W: int, O: int, kernel_size: int, stride: int, padding: int,
                             dilation: int) -> int:
    return int(_c_w8_ws(B, C, H, W, O, kernel_size, stride, padding, dilation))


def bt_w8a8_conv2d(x: torch.Tensor, w: torch.Tensor, stride: int, padding: int, dilation: int, smooth: bool = False,
                   out_dtype=torch.float32, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """W8A8 im2col + gemm convolution of NCHW x with OIHW w (f32 or bf16),
    optionally with SmoothQuant; NCHW out in out_dtype (f32 or bf16)."""
    _contig(x, "x")
    _contig(w, "w")
    B, C, H, W = x.shape
    O, _, k, _ = w.shape
    Ho, Wo = conv2d_out_size(H, k, stride, padding, dilation), conv2d_out_size(W, k, stride, padding, dilation)
    if out is None:
        out = torch.empty((B, O, max(Ho, 0), max(Wo, 0)), dtype=out_dtype, device=x.device)
    ws = _workspace(bt_w8a8_conv2d_workspace(B, C, H, W, O, k, stride, padding, dilation), x.device, workspace)
    _check(_c_w8(_ptr(x), _DT[x.dtype], _ptr(w), _DT[w.dtype], B, C, H, W, O, k, stride, padding, dilation,
                 1 if smooth else 0, _ptr(out), _DT[out.dtype], _ptr(ws), 0 if ws is None else ws.numel(),
                 _stream(stream)))
    return out


def bt_scale_init(x: torch.Tensor, factor: float = 2.0, scale_dtype=None, out: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """(factor * x.abs().mean()).to(scale_dtype) computed on the device into a
    one-element float tensor (scale_dtype defaults to x's dtype)."""
    _contig(x, "x")
    if out is None:
        out = torch.empty(1, dtype=torch.float32, device=x.device)
    st = _DT[x.dtype if scale_dtype is None else scale_dtype]
    _check(_c_scale_init(_ptr(x), _DT[x.dtype], x.numel(), factor, st, _ptr(out), _stream(stream)))
    return out


def bt_binary_linear_noalloc_max_bytes() -> int:
    return int(_c_noalloc_max())


def bt_binary_linear_noalloc(x: torch.Tensor, weight: torch.Tensor, w_code: int, K: int, scale_a: float,
                             scale_w: float, bias_a=None, out_dtype=None, algo: int = BT_ALGO_AUTO,
                             x_packed: bool = False, out: torch.Tensor | None = None,
                             stream=None) -> torch.Tensor:
    """bt_binary_linear without a workspace: for callers that cannot allocate
    device memory (the packed activations go to the library's fixed scratch
    array). Only `out`, if not given, is allocated here, by torch."""
    _contig(x, "x")
    _contig(weight, "weight")
    M, N = x.shape[0], weight.shape[0]
    xt = BT_PACKED if x_packed else _DT[x.dtype]
    if out_dtype is None:
        out_dtype = x.dtype if not x_packed else torch.float32
    ot = _DT[out_dtype]
    if out is None:
        out = torch.empty((M, N), dtype=_TORCH[ot], device=x.device)
    blen = 0 if bias_a is None else bias_a.numel()
    _check(_c_lin_noalloc(_ptr(x), xt, _ptr(weight), w_code, M, N, K, scale_a, scale_w, _ptr(bias_a), blen,
                          _ptr(out), ot, algo, _stream(stream)))
    return out


def bt_plan(op: int, M: int, N: int, K: int) -> tuple[int, int]:
    """The (code, algo) the library runs fastest for this problem size."""
    code, algo = _i(0), _i(0)
    _check(_c_plan(op, M, N, K, ctypes.byref(code), ctypes.byref(algo)))
    return code.value, algo.value


def bt_tune_linear(x: torch.Tensor, weight: torch.Tensor, w_code: int, K: int, scale_a: float, scale_w: float,
                   bias_a=None, out_dtype=None, x_packed: bool = False, reps: int = 10,
                   out: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None) -> dict:
    """Time this linear forward in every candidate launch shape and keep the
    fastest for later bt_binary_linear calls of the same size; returns the
    bt_tune_result fields as a dict."""
    _contig(x, "x")
    _contig(weight, "weight")
    M, N = x.shape[0], weight.shape[0]
    xt = BT_PACKED if x_packed else _DT[x.dtype]
    if out_dtype is None:
        out_dtype = x.dtype if not x_packed else torch.float32
    ot = _DT[out_dtype]
    if out is None:
        out = torch.empty((M, N), dtype=_TORCH[ot], device=x.device)
    ws = _workspace(bt_binary_linear_workspace(M, K, xt, w_code), x.device, workspace)
    blen = 0 if bias_a is None else bias_a.numel()
    res = TuneResult()
    _check(_c_tune(_ptr(x), xt, _ptr(weight), w_code, M, N, K, scale_a, scale_w, _ptr(bias_a), blen, _ptr(out), ot,
                   _ptr(ws), 0 if ws is None else ws.numel(), reps, _stream(stream), ctypes.byref(res)))
    return {f: getattr(res, f) for f, _ in TuneResult._fields_}


def bt_tune_conv2d(x: torch.Tensor, weight: torch.Tensor, w_code: int, C: int, kernel_size: int, stride: int,
                   padding: int, dilation: int, scale_a: float, scale_w: float, bias_a=None, out_dtype=None,
                   x_packed: bool = False, reps: int = 10, out: torch.Tensor | None = None,
                   workspace: torch.Tensor | None = None, stream=None) -> dict:
    """Time this convolution in every candidate plan and keep the fastest for
    later bt_binary_conv2d calls of the same geometry; returns the
    bt_tune_conv_result fields as a dict."""
    _contig(x, "x")
    _contig(weight, "weight")
    if x_packed:
        B, H, W = x.shape[0], x.shape[1], x.shape[2]
        xt = BT_PACKED
    else:
        B, C2, H, W = x.shape
        if C2 != C:
            raise ValueError("C does not match x")
        xt = _DT[x.dtype]
    O = weight.shape[0]
    if out_dtype is None:
        out_dtype = x.dtype if not x_packed else torch.float32
    ot = _DT[out_dtype]
    Ho = conv2d_out_size(H, kernel_size, stride, padding, dilation)
    Wo = conv2d_out_size(W, kernel_size, stride, padding, dilation)
    if out is None:
        out = torch.empty((B, O, max(Ho, 0), max(Wo, 0)), dtype=_TORCH[ot], device=x.device)
    ws = _workspace(bt_binary_conv2d_workspace(B, C, H, W, kernel_size, stride, padding, dilation, xt, w_code),
                    x.device, workspace)
    blen = 0 if bias_a is None else bias_a.numel()
    res = TuneConvResult()
    _check(_c_tune_conv(_ptr(x), xt, _ptr(weight), w_code, B, C, H, W, O, kernel_size, stride, padding, dilation,
                        scale_a, scale_w, _ptr(bias_a), blen, _ptr(out), ot, _ptr(ws), 0 if ws is None else ws.numel(),
                        reps, _stream(stream), ctypes.byref(res)))
    return {f: getattr(res, f) for f, _ in TuneConvResult._fields_}


class ConvPlanInfo(ctypes.Structure):
    """bt_conv_plan_info: the tiling of the implicit-im2col convolution."""
    _fields_ = [(n, _i) for n in ("implicit", "pair", "weights_resident", "pixel_stages", "bands", "band_rows",
                                  "cta_rows", "row_width", "tile_n", "cta_n", "staged_rows", "phases",
                                  "max_tap_shift", "tiles", "smem_bytes")]


_c_plan_info = _sig("bt_conv2d_plan_info", _i, [_i64, _i64, _i64, _i64, _i64, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                               ctypes.POINTER(ConvPlanInfo)])


def bt_conv2d_plan_info(B: int, C: int, H: int, W: int, O: int, kernel_size: int, stride: int, padding: int,
                        dilation: int, code: int, out_dtype=torch.float32, sms: int = 152, pair: int = -1,
                        split: int = 1) -> dict:
    """The tiling the implicit-im2col convolution takes for this geometry
    (host only): the bt_conv_plan_info fields as a dict."""
    info = ConvPlanInfo()
    _check(_c_plan_info(B, C, H, W, O, kernel_size, stride, padding, dilation, code, _DT[out_dtype], sms, pair,
                        split, ctypes.byref(info)))
    return {f: getattr(info, f) for f, _ in ConvPlanInfo._fields_}


def bt_tune_reset() -> None:
    """Forget every launch shape, plan and code bt_tune_linear / bt_tune_conv2d kept."""
    _c_tune_reset()


def bt_set_wait_timeout(ns: int) -> None:
    """Limit (ns) of the tensor-core kernels' bounded waits for later launches;
    0 restores the default (2 s)."""
    _check(_c_wait(ns))


def bt_device_status(stream=None) -> int:
    """Synchronize the stream; return (and clear) the device error status."""
    return int(_c_status(_stream(stream)))
