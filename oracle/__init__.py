"""CPU oracle for the binarized linear / conv2d forward.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The library under
``xnor_popcount_gemm_gb300`` never imports it, and this package imports
nothing from there: the two share no code.

The nested loops live in ``bt_oracle.c`` (plain C, compiled here with gcc);
this module binarizes and contracts through them and does the epilogue with
plain numpy / PyTorch CPU ops. Every function cites the passage it follows:

* bitorch-engine ``BinaryConv2dCutlass.set_activation``: the activation shift
  ``x + bias_a`` before binarizing ("learnable shift input").
* bitorch-engine ``BinaryConv2dForward.forward``: the native forward is given
  ``scale_a.item() * scale_w.item()`` and its result is cast back with
  ``out.to(x.dtype)``.
* bitorch-engine ``BinaryLinearForward.forward``: "the result of the binary
  linear operation scaled by the activation and weight scaling factors".
* banghao.live/blog/9, section 2 (``MyConv2d.forward``): the output-size
  formula and the unfold + mm lowering of a convolution.
* torch/ao/quantization/experimental/linear.py, ``LinearAPoT.matmul``: the
  plain i-j-k triple loop of a matrix product.
* banghao.live/blog/9, sections 3 and 4 (``MyQuantConv2d.forward``): the
  W8A8 im2col + gemm convolution, with and without the SmoothQuant per-column
  scale migration ``scale = sqrt(act_max / weight_max)``.
* bitorch-engine ``BinaryConv2dForward.backward`` (the straight-through
  backward written out in code) and ``BinaryLinearForward.backward`` (the
  same steps in prose for the linear layer): ``grad_input`` from the upstream
  gradient and ``sign(w) * scale_w`` in the gradient's dtype, zeroed where
  ``x / scale_a`` falls outside [-1, 1]; ``grad_scale_a`` as the sum of
  ``grad_input * sign(x) / sqrt(numel)``; ``grad_weight`` from
  ``sign(x) * scale_a`` and the upstream gradient. (The int8 quantization of
  ``grad_weight`` that follows on the page is not part of this oracle.)

Readings where the sources leave a step open:

1. The binarization threshold: ``x + bias >= 0`` gives +1, anything else
   (negative, NaN) gives -1; -0.0 gives +1. Weights are binarized with the
   same rule and no shift. The sum is taken in double, so its sign is the
   sign of the exact sum.
2. A positive ``scale_a`` does not change a sign, so the division by
   ``scale_a`` of "integrated scaling and value range conversion" is not
   applied before the threshold.
3. The native call receives one float ``alpha = fp32(scale_a * scale_w)``
   (the double product of two floats, rounded once to float); the native
   result is ``fp32(dot * alpha)`` (one rounding) and ``.to(x.dtype)`` then
   rounds to nearest-even.
4. A convolution tap in the zero padding contributes 0 to the dot product,
   as in the unfold + mm lowering.
5. Backward: the page's steps; for the linear layer with the convolution's
   input and weight gradients replaced by the two matrix products
   ``g @ wt`` and ``g^T @ xs``. Each product is formed exactly (double) and
   rounded once to the gradient's dtype (bf16), as a matrix product in that
   dtype returns it; ``x / scale_a`` is an fp32 division rounded to x's
   dtype before the comparison with -1 and 1; ``grad_input`` is the
   rounded product times the fp32 mask (so fp32, holding bf16 values); the
   ``grad_scale_a`` terms are fp32 products and their sum is taken in double.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch
import torch.nn.functional as F

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bt_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``bt_oracle.c`` into ``_build/liboracle.so`` (gcc, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.orc_binarize.argtypes = [p, i64, p, i64, i64, p]
        lib.orc_linear_dot.argtypes = [p, p, i64, i64, i64, p]
        lib.orc_linear_dot_at.argtypes = [p, p, i64, p, p, i64, p]
        lib.orc_conv2d_dot.argtypes = [p, p] + [i64] * 9 + [p]
        lib.orc_conv2d_dot_at.argtypes = [p, p] + [i64] * 9 + [p, i64, p]
        lib.orc_conv2d_out_size.argtypes = [i64] * 5
        lib.orc_conv2d_out_size.restype = i64
        for f in ("orc_binarize", "orc_linear_dot", "orc_linear_dot_at", "orc_conv2d_dot",
                  "orc_conv2d_dot_at"):
            getattr(lib, f).restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _as_f32(x) -> np.ndarray:
    """Exact conversion of an fp32 / bf16 / fp16 tensor or array to fp32 numpy."""
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu()
        if x.dtype not in (torch.float32, torch.bfloat16, torch.float16):
            raise TypeError(f"unsupported dtype {x.dtype}")
        return np.ascontiguousarray(x.to(torch.float32).numpy())
    x = np.asarray(x)
    if x.dtype not in (np.float32, np.float16):
        raise TypeError(f"unsupported dtype {x.dtype}")
    return np.ascontiguousarray(x.astype(np.float32))


# ----------------------------------------------------------------------------
# Binarization (set_activation's shift, then the sign threshold)
# ----------------------------------------------------------------------------

def binarize(x, bias=None, channel_axis: int | None = None) -> np.ndarray:
    """+1/-1 int8 array: ``+1`` where ``x + bias >= 0`` (sum in double), else -1.

    ``bias`` is None (no shift), a scalar, or a 1-D array along
    ``channel_axis`` (the per-channel ``bias_a.view(1,-1,1,1)`` of
    ``BinaryConv2dCutlass.set_activation`` uses ``channel_axis=1``; the
    layer-wise bias of ``BinaryLinearCuda`` is a scalar).
    """
    xf = _as_f32(x)
    out = np.empty(xf.shape, dtype=np.int8)
    if bias is None:
        b = np.zeros(1, np.float32)
        blen, inner = 0, 1
    else:
        b = np.ascontiguousarray(_as_f32(bias).reshape(-1))
        if b.size == 1:
            blen, inner = 1, 1
        else:
            if channel_axis is None:
                raise ValueError("a vector bias needs channel_axis")
            ax = channel_axis % xf.ndim
            if xf.shape[ax] != b.size:
                raise ValueError("bias length does not match the channel axis")
            blen = b.size
            inner = int(np.prod(xf.shape[ax + 1:], dtype=np.int64))
    _load().orc_binarize(_ptr(xf), xf.size, _ptr(b), blen, inner, _ptr(out))
    return out


def binarize_weight(w) -> np.ndarray:
    """Weights: +1 where ``w >= 0``, else -1 (no shift)."""
    return binarize(w)


# ----------------------------------------------------------------------------
# Contractions (nested loops in C)
# ----------------------------------------------------------------------------

def linear_dot(sa: np.ndarray, sw: np.ndarray) -> np.ndarray:
    """``dot[m,n] = sum_k sa[m,k] sw[n,k]`` as int32 (the i-j-k loop)."""
    sa = np.ascontiguousarray(sa, dtype=np.int8)
    sw = np.ascontiguousarray(sw, dtype=np.int8)
    M, K = sa.shape
    N, K2 = sw.shape
    if K != K2:
        raise ValueError("K mismatch")
    dot = np.empty((M, N), dtype=np.int32)
    _load().orc_linear_dot(_ptr(sa), _ptr(sw), M, N, K, _ptr(dot))
    return dot


def linear_dot_at(sa: np.ndarray, sw: np.ndarray, rows, cols) -> np.ndarray:
    """The same sums for the listed (row, col) pairs only."""
    sa = np.ascontiguousarray(sa, dtype=np.int8)
    sw = np.ascontiguousarray(sw, dtype=np.int8)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if sa.shape[1] != sw.shape[1] or rows.shape != cols.shape:
        raise ValueError("shape mismatch")
    out = np.empty(rows.shape, dtype=np.int32)
    _load().orc_linear_dot_at(_ptr(sa), _ptr(sw), sa.shape[1], _ptr(rows), _ptr(cols),
                              rows.size, _ptr(out))
    return out


def conv2d_out_size(h: int, k: int, s: int, p: int, d: int) -> int:
    """``floor((h + 2p - d(k-1) - 1)/s + 1)`` (banghao.live/blog/9, section 2);
    0 when the window does not fit."""
    return int(_load().orc_conv2d_out_size(h, k, s, p, d))


def conv2d_dot(sa: np.ndarray, sw: np.ndarray, stride: int, padding: int, dilation: int) -> np.ndarray:
    """Direct 7-loop convolution of +1/-1 NCHW ``sa`` with OIHW ``sw``; padded taps add 0."""
    sa = np.ascontiguousarray(sa, dtype=np.int8)
    sw = np.ascontiguousarray(sw, dtype=np.int8)
    B, C, H, W = sa.shape
    O, C2, k, k2 = sw.shape
    if C != C2 or k != k2:
        raise ValueError("shape mismatch")
    Ho = conv2d_out_size(H, k, stride, padding, dilation)
    Wo = conv2d_out_size(W, k, stride, padding, dilation)
    dot = np.empty((B, O, Ho, Wo), dtype=np.int32)
    if dot.size:
        _load().orc_conv2d_dot(_ptr(sa), _ptr(sw), B, C, H, W, O, k, stride, padding, dilation,
                               _ptr(dot))
    return dot


def conv2d_dot_at(sa: np.ndarray, sw: np.ndarray, stride: int, padding: int, dilation: int,
                  flat_index) -> np.ndarray:
    """The same sums at the listed flat indices of the NCHW output only."""
    sa = np.ascontiguousarray(sa, dtype=np.int8)
    sw = np.ascontiguousarray(sw, dtype=np.int8)
    B, C, H, W = sa.shape
    O, _, k, _ = sw.shape
    idx = np.ascontiguousarray(flat_index, dtype=np.int64)
    out = np.empty(idx.shape, dtype=np.int32)
    _load().orc_conv2d_dot_at(_ptr(sa), _ptr(sw), B, C, H, W, O, k, stride, padding, dilation,
                              _ptr(idx), idx.size, _ptr(out))
    return out


# ----------------------------------------------------------------------------
# Epilogue: alpha = scale_a * scale_w, fp32 result, cast to the output dtype
# ----------------------------------------------------------------------------

_TORCH_OUT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16, "i32": torch.int32}


def alpha(scale_a: float, scale_w: float) -> np.float32:
    """``fp32(scale_a * scale_w)``: the double product of the two float scales
    (``scale_a.item()*scale_w.item()``) rounded once to float."""
    a = np.float64(np.float32(scale_a))
    w = np.float64(np.float32(scale_w))
    return np.float32(a * w)


def epilogue(dot: np.ndarray, scale_a: float, scale_w: float, out_dtype: str) -> torch.Tensor:
    """``fp32(dot * alpha)`` (exact product in double, one rounding to float),
    then ``.to(out_dtype)`` (round to nearest even). ``i32`` returns ``dot``."""
    dot = np.asarray(dot, dtype=np.int32)
    if out_dtype == "i32":
        return torch.from_numpy(dot.copy())
    al = np.float64(alpha(scale_a, scale_w))
    y64 = dot.astype(np.float64) * al          # exact: 24-bit integer times 24-bit float
    y32 = torch.from_numpy(y64.astype(np.float32))
    return y32.to(_TORCH_OUT[out_dtype])


def binary_linear(x, w, scale_a: float, scale_w: float, bias_a=None, out_dtype: str = "f32"):
    """Whole linear forward: shift + sign, sign of W, contraction, epilogue."""
    sa = binarize(x, bias_a, channel_axis=-1)
    sw = binarize_weight(w)
    return epilogue(linear_dot(sa, sw), scale_a, scale_w, out_dtype)


def binary_conv2d(x, w, scale_a: float, scale_w: float, stride: int, padding: int, dilation: int,
                  bias_a=None, out_dtype: str = "f32"):
    """Whole conv2d forward (NCHW in, OIHW weights, NCHW out)."""
    sa = binarize(x, bias_a, channel_axis=1)
    sw = binarize_weight(w)
    return epilogue(conv2d_dot(sa, sw, stride, padding, dilation), scale_a, scale_w, out_dtype)


# ----------------------------------------------------------------------------
# The packed operand formats the library documents, written out plainly so the
# packing kernels can be checked bit for bit.
# ----------------------------------------------------------------------------

CODE_BITS, CODE_E4M3, CODE_E2M1 = 0, 1, 2


def packed_row_bytes(k: int, code: int) -> int:
    """Bytes per packed row of ``k`` elements: BITS rows rounded up to 16
    bytes, E4M3 / E2M1 rows to 64 bytes."""
    if code == CODE_BITS:
        return (((k + 31) // 32) * 4 + 15) // 16 * 16
    if code == CODE_E4M3:
        return (k + 63) // 64 * 64
    if code == CODE_E2M1:
        return ((k + 1) // 2 + 63) // 64 * 64
    raise ValueError(code)


def pack_rows(s: np.ndarray, code: int) -> np.ndarray:
    """Pack the last axis of a +1/-1 array into the documented format.

    BITS: uint32 words, bit j of word w holds element 32w + j, 1 for +1.
    E4M3: one byte per element, 0x38 (+1.0) or 0xB8 (-1.0).
    E2M1: two elements per byte, element 2i in the low nibble; 0x2 (+1.0) or
    0xA (-1.0). Every position past the last element, up to the padded row
    length, is 0. Returns uint8 [..., packed_row_bytes].
    """
    s = np.asarray(s, dtype=np.int8)
    lead, k = s.shape[:-1], s.shape[-1]
    rows = s.reshape(-1, k)
    nb = packed_row_bytes(k, code)
    out = np.zeros((rows.shape[0], nb), dtype=np.uint8)
    if code == CODE_BITS:
        words = out.view(np.uint32)
        for kk in range(k):
            bit = (rows[:, kk] > 0).astype(np.uint32) << np.uint32(kk % 32)
            words[:, kk // 32] |= bit
    elif code == CODE_E4M3:
        out[:, :k] = np.where(rows > 0, 0x38, 0xB8).astype(np.uint8)
    else:
        nib = np.where(rows > 0, 0x2, 0xA).astype(np.uint8)
        for kk in range(k):
            shift = 4 * (kk % 2)
            out[:, kk // 2] |= (nib[:, kk] << shift).astype(np.uint8)
    return out.reshape(*lead, nb)


def pack_nchw_to_nhwc(s: np.ndarray, code: int) -> np.ndarray:
    """Channel-packed NHWC: [B,C,H,W] +1/-1 -> uint8 [B,H,W,packed_row_bytes(C)].

    Also the conv weight format: OIHW [O,C,k,k] -> [O,k,k,packed_row_bytes(C)].
    """
    s = np.asarray(s, dtype=np.int8)
    return pack_rows(np.ascontiguousarray(np.transpose(s, (0, 2, 3, 1))), code)


# ----------------------------------------------------------------------------
# Backward (straight-through estimator) of the binary linear layer, following
# bitorch-engine BinaryConv2dForward.backward step by step with the conv
# gradients replaced by matrix products (BinaryLinearForward.backward states
# the same steps for the linear layer).
# ----------------------------------------------------------------------------

_BF16_MAX = float.fromhex("0x1.fep127")


def bf16_round(a) -> np.ndarray:
    """Round to the nearest bfloat16 value, ties to even, from float64 (one
    rounding); returns float32 holding bf16 values. NaN stays NaN, values
    beyond the largest finite bf16 after rounding become +-inf."""
    v = np.asarray(a, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.float64)
    fin = np.isfinite(v)
    out[~fin] = v[~fin]
    vf = v[fin]
    _, e = np.frexp(vf)                       # vf = m * 2**e, 0.5 <= |m| < 1
    # 8 significant bits: the spacing is 2**(e-8); below the normal range
    # (e - 1 < -126) the spacing stays 2**-133
    step = np.ldexp(1.0, np.maximum(e, -125) - 8)
    r = np.rint(vf / step) * step             # rint rounds half to even
    r[np.abs(r) > _BF16_MAX] = np.inf * np.sign(r[np.abs(r) > _BF16_MAX])
    out[fin] = r
    return out.astype(np.float32)


def sign(a) -> np.ndarray:
    """``torch.sign``, which is ``(a > 0) - (a < 0)``: -1, 0 or +1, and 0 for
    NaN and for -0.0."""
    a = np.asarray(a, dtype=np.float32)
    return ((a > 0).astype(np.float32) - (a < 0).astype(np.float32)).astype(np.float32)


def linear_backward(x, w, g, scale_a: float, scale_w: float, x_dtype: str = "bf16") -> dict:
    """The three gradients of the binary linear layer for upstream gradient
    ``g`` [M, N] (bf16 values), input ``x`` [M, K], weight ``w`` [N, K].

    Steps (BinaryConv2dForward.backward):
      wt = (sign(w) in g's dtype) * scale_w        -> bf16(sign(w) * scale_w)
      grad_input = g @ wt                          -> exact sum, rounded to bf16
      q = x / scale_a (x's dtype); middle = 1 - [q < -1] - [q > 1]
      grad_input = grad_input * middle             (fp32)
      grad_scale_a = sum(grad_input * sign(x) * (1 / sqrt(numel(x))))
      grad_weight = g^T @ (sign(x) * scale_a)      -> exact sum, rounded to bf16
    Returns the rounded and the exact (float64) products as well."""
    x32 = _as_f32(x)
    w32 = _as_f32(w)
    g64 = _as_f32(g).astype(np.float64)
    M, K = x32.shape
    sa32, sw32 = np.float32(scale_a), np.float32(scale_w)
    wt = bf16_round(sign(w32) * sw32)                       # [N, K]
    gi_exact = g64 @ wt.astype(np.float64)                  # [M, K]
    gi = bf16_round(gi_exact)
    q = x32 / sa32                                          # fp32 division
    if x_dtype in ("bf16",):
        q = bf16_round(q)
    elif x_dtype == "f16":
        q = torch.from_numpy(q).to(torch.float16).float().numpy()
    middle = (1.0 - (q < -1).astype(np.float32) - (q > 1).astype(np.float32)).astype(np.float32)
    grad_input = (gi * middle).astype(np.float32)
    inv = np.float32(1.0 / np.sqrt(np.float64(M * K)))
    terms = ((grad_input * sign(x32)).astype(np.float32) * inv).astype(np.float32)
    grad_scale_a = float(terms.astype(np.float64).sum())
    xs = bf16_round(sign(x32) * sa32)                       # [M, K]
    gw_exact = g64.T @ xs.astype(np.float64)                # [N, K]
    return {"grad_input": grad_input, "grad_input_exact": gi_exact, "middle": middle,
            "grad_scale_a": grad_scale_a, "grad_scale_a_abs": float(np.abs(terms.astype(np.float64)).sum()),
            "grad_weight": bf16_round(gw_exact), "grad_weight_exact": gw_exact}


def conv2d_backward(x, w, g, scale_a: float, scale_w: float, stride: int, padding: int, dilation: int,
                    x_dtype: str = "bf16") -> dict:
    """The three gradients of the binary conv2d layer (BinaryConv2dForward.backward)
    for upstream gradient ``g`` [B, O, Ho, Wo] (bf16 values), input ``x``
    [B, C, H, W], weight ``w`` [O, C, k, k]:
      wt = bf16(sign(w) * scale_w)
      grad_input = conv2d_input(x.shape, wt, g)    -> exact, rounded to bf16
      q = x / scale_a (x's dtype); grad_input *= 1 - [q < -1] - [q > 1]
      grad_scale_a = sum(grad_input * sign(x) * (1 / sqrt(numel(x))))
      grad_weight = conv2d_weight(bf16(sign(x) * scale_a), w.shape, g) -> exact, rounded to bf16
    The two convolution gradients are torch.nn.grad's routines in float64
    (the page calls the same two routines), exact for these operands."""
    x32 = _as_f32(x)
    w32 = _as_f32(w)
    g64 = torch.from_numpy(_as_f32(g).astype(np.float64))
    B, C, H, W = x32.shape
    sa32, sw32 = np.float32(scale_a), np.float32(scale_w)
    wt = torch.from_numpy(bf16_round(sign(w32) * sw32).astype(np.float64))
    gi_exact = torch.nn.grad.conv2d_input((B, C, H, W), wt, g64, stride=stride, padding=padding,
                                          dilation=dilation).numpy()
    gi = bf16_round(gi_exact)
    q = x32 / sa32
    if x_dtype == "bf16":
        q = bf16_round(q)
    elif x_dtype == "f16":
        q = torch.from_numpy(q).to(torch.float16).float().numpy()
    middle = (1.0 - (q < -1).astype(np.float32) - (q > 1).astype(np.float32)).astype(np.float32)
    grad_input = (gi * middle).astype(np.float32)
    inv = np.float32(1.0 / np.sqrt(np.float64(x32.size)))
    terms = ((grad_input * sign(x32)).astype(np.float32) * inv).astype(np.float32)
    xs = torch.from_numpy(bf16_round(sign(x32) * sa32).astype(np.float64))
    gw_exact = torch.nn.grad.conv2d_weight(xs, tuple(w32.shape), g64, stride=stride, padding=padding,
                                           dilation=dilation).numpy()
    return {"grad_input": grad_input, "grad_input_exact": gi_exact, "middle": middle,
            "grad_scale_a": float(terms.astype(np.float64).sum()),
            "grad_scale_a_abs": float(np.abs(terms.astype(np.float64)).sum()),
            "grad_weight": bf16_round(gw_exact), "grad_weight_exact": gw_exact}


def conv2d_grad_weight_at(x, g, scale_a: float, stride: int, padding: int, dilation: int, k: int, o_idx,
                          t_idx) -> np.ndarray:
    """Entries (o, t) of conv2d_backward's exact weight gradient, t = (c, kh,
    kw) flattened in OIHW order: the sum over images b and output pixels
    (i, j) of g[b, o, i, j] * bf16(sign(x) * scale_a)[b, c, i*s - p + kh*d,
    j*s - p + kw*d] (0 in the padding), in float64, from the unfold of the
    scaled signs. For layers whose whole gradient is too slow here."""
    x32 = _as_f32(x)
    g64 = _as_f32(g).astype(np.float64)
    xs = torch.from_numpy(bf16_round(sign(x32) * np.float32(scale_a)).astype(np.float64))
    u = F.unfold(xs, k, dilation=dilation, padding=padding, stride=stride).numpy()     # [B, C*k*k, L]
    gl = g64.reshape(g64.shape[0], g64.shape[1], -1)                                 # [B, O, L]
    o_idx, t_idx = np.asarray(o_idx), np.asarray(t_idx)
    out = np.empty(o_idx.size, np.float64)
    for s0 in range(0, o_idx.size, 64):
        o, t = o_idx[s0:s0 + 64], t_idx[s0:s0 + 64]
        out[s0:s0 + 64] = (gl[:, o, :] * u[:, t, :]).sum(axis=(0, 2))
    return out


def scale_init(x, factor: float, x_dtype: str, scale_dtype: str) -> float:
    """BinaryConv2dCutlass.set_activation's first-call scale:
    (factor * x.abs().mean()).to(layer dtype). Reading: the mean is the exact
    sum of |x| (float64) divided by n (one double division), rounded once to
    x's dtype (x.abs().mean() is a tensor of x's dtype); factor * mean is
    rounded to x's dtype, then to the layer's dtype."""
    def to(v, dt):
        v = np.asarray(v, dtype=np.float64)
        if dt == "bf16":
            return float(bf16_round(v))
        if dt == "f16":
            return float(torch.tensor(float(v), dtype=torch.float64).to(torch.float16).item())
        return float(np.float32(v))
    a = np.abs(_as_f32(x).astype(np.float64))
    mean = to(a.sum() / a.size, x_dtype)
    return to(to(np.float64(factor) * mean, x_dtype), scale_dtype)


# ----------------------------------------------------------------------------
# W8A8 im2col + gemm convolution (banghao.live/blog/9 sections 3 and 4)
# ----------------------------------------------------------------------------

def fake_quant_int8(v: np.ndarray):
    """The quantizers the page applies to the im2col rows and the flattened
    weights, read as per-tensor symmetric int8 on [-127, 127] with a dynamic
    max: amax = max|v|, scale = fp32(amax / 127), q = clamp(round-half-even(
    v * fp32(1 / scale)), -127, 127) (torch's fake-quant rounding); returns q
    (int64) and scale. An all-zero tensor gives q = 0, scale = 0."""
    v = np.asarray(v, dtype=np.float32)
    amax = np.float32(np.abs(v).max()) if v.size else np.float32(0)
    if amax == 0:
        return np.zeros(v.shape, np.int64), np.float32(0)
    scale = np.float32(amax / np.float32(127))
    inv = np.float32(np.float32(1) / scale)
    q = np.clip(np.rint((v * inv).astype(np.float32)), -127, 127).astype(np.int64)
    return q, scale


def _w8a8_quantized(x, w, stride: int, padding: int, dilation: int, smooth: bool):
    """The quantized operands of MyQuantConv2d.forward (see w8a8_conv2d):
    returns (rows, wf, scale_col, qx, sx, qw, sw, alpha, (B, O, ho, wo))."""
    x32 = torch.from_numpy(_as_f32(x))
    w32 = _as_f32(w)
    B, C, H, W = x32.shape
    O, _, k, _ = w32.shape
    ho = conv2d_out_size(H, k, stride, padding, dilation)
    wo = conv2d_out_size(W, k, stride, padding, dilation)
    rows = F.unfold(x32, k, dilation=dilation, padding=padding, stride=stride)     # [B, C*k*k, L]
    rows = rows.transpose(1, 2).reshape(-1, C * k * k).numpy().astype(np.float32)
    wf = w32.reshape(O, C * k * k).astype(np.float32)
    scale_col = None
    if smooth:
        act = np.abs(rows).max(axis=0).astype(np.float32)
        wmax = np.abs(wf).max(axis=0).astype(np.float32)
        with np.errstate(divide="ignore", invalid="ignore"):
            scale_col = np.sqrt((act / wmax).astype(np.float32)).astype(np.float32)
            rows = (rows / scale_col).astype(np.float32)
            wf = (wf * scale_col).astype(np.float32)
    qx, sx = fake_quant_int8(rows)
    qw, sw = fake_quant_int8(wf)
    alpha = np.float32(np.float64(sx) * np.float64(sw))
    return rows, wf, scale_col, qx, sx, qw, sw, alpha, (B, O, ho, wo)


def w8a8_conv2d(x, w, stride: int, padding: int, dilation: int, smooth: bool = False) -> dict:
    """MyQuantConv2d.forward: unfold x into im2col rows [P, C*k*k] (zero
    padding), flatten w to [O, C*k*k]; with SmoothQuant, per column
    act = max|rows|, wmax = max|w|, scale = sqrt(act / wmax) (fp32), rows /=
    scale, w *= scale; quantize both (fake_quant_int8); the product of the
    dequantized values is sum(q_x * q_w) * s_x * s_w, taken exactly and
    rounded as y = fp32(double(dot) * double(fp32(s_x * s_w))); NCHW out."""
    rows, wf, scale_col, qx, sx, qw, sw, alpha, (B, O, ho, wo) = _w8a8_quantized(x, w, stride, padding, dilation,
                                                                                 smooth)
    dot = qx @ qw.T                                                                # exact int64 [P, O]
    y = (dot.astype(np.float64) * np.float64(alpha)).astype(np.float32)
    y = y.reshape(B, ho * wo, O).transpose(0, 2, 1).reshape(B, O, ho, wo)
    return {"y": np.ascontiguousarray(y), "dot": dot, "qx": qx, "qw": qw, "sx": sx, "sw": sw, "alpha": alpha,
            "scale": scale_col, "rows": rows, "wf": wf}


def w8a8_conv2d_at(x, w, stride: int, padding: int, dilation: int, smooth: bool, flat) -> np.ndarray:
    """w8a8_conv2d's output at the flat NCHW indices `flat` only: the maxima
    and the quantization over every row as there, the dot products of the
    requested outputs alone (for workloads whose full product is too slow)."""
    _, _, _, qx, _, qw, _, alpha, (B, O, ho, wo) = _w8a8_quantized(x, w, stride, padding, dilation, smooth)
    flat = np.asarray(flat, dtype=np.int64)
    j = flat % wo
    i = (flat // wo) % ho
    o = (flat // (wo * ho)) % O
    b = flat // (wo * ho * O)
    p = (b * ho + i) * wo + j
    dot = np.einsum("ij,ij->i", qx[p], qw[o])
    return (dot.astype(np.float64) * np.float64(alpha)).astype(np.float32)