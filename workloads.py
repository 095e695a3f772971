"""Seeded synthetic workloads for the binarized linear / conv2d forward.

This module only draws inputs. It holds none of the method's arithmetic, and
both the CPU oracle (through the tests and the benchmark) and the CUDA library
receive exactly the tensors it returns.

Recipe, for every workload: values are drawn in fp32 on the CPU with a
``torch.Generator`` seeded per workload, then cast with ``.to(bfloat16)``
where the workload is bf16. Scales are ``mean|.|`` of the cast tensor,
reduced in float64 and rounded once to fp32. A scalar activation bias, where
one is used, is drawn from U(-0.1, 0.1) in fp32.

The shapes are those of the binarized layers bitorch-engine and the
im2col+gemm write-up deal with: a small linear, an
LLM projection (4096 x 4096), ResNet-style 3x3 convolutions (stride 1; stride
2 with dilation 1 and 2), and a large linear plus one with ragged M, N, K.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass
class Workload:
    name: str
    kind: str                 # "linear" or "conv"
    x: torch.Tensor           # [M,K] or NCHW [B,C,H,W]
    w: torch.Tensor           # [N,K] or OIHW [O,C,k,k]
    scale_a: float
    scale_w: float
    bias: torch.Tensor | None  # fp32, shape [1] (scalar) or [C]; None for no shift
    out_dtype: str            # "f32" or "bf16"
    stride: int = 1
    padding: int = 0
    dilation: int = 1
    meta: dict = field(default_factory=dict)

    @property
    def x_dtype(self) -> str:
        return {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}[self.x.dtype]

    def gemm_shape(self) -> tuple[int, int, int]:
        """(M, N, K) of the contraction; for a conv, M = B*Ho*Wo, N = O, K = C*k*k."""
        if self.kind == "linear":
            return self.x.shape[0], self.w.shape[0], self.x.shape[1]
        B, C, H, W = self.x.shape
        O, _, k, _ = self.w.shape
        ho = (H + 2 * self.padding - self.dilation * (k - 1) - 1) // self.stride + 1
        wo = (W + 2 * self.padding - self.dilation * (k - 1) - 1) // self.stride + 1
        return B * ho * wo, O, C * k * k

    def binary_ops(self) -> int:
        m, n, k = self.gemm_shape()
        return 2 * m * n * k


def mean_abs(t: torch.Tensor) -> float:
    """mean |t| reduced in float64, rounded once to fp32."""
    v = t.detach().to(torch.float64).abs().mean().item()
    return float(torch.tensor(v, dtype=torch.float64).to(torch.float32).item())


def _normal(gen, shape, std=1.0):
    return torch.randn(*shape, generator=gen, dtype=torch.float32) * std


def _cast(t, dtype):
    return t.to(dtype) if dtype != torch.float32 else t


def linear(name, M, N, K, *, dtype=torch.float32, w_std=1.0, bias="none", seed=0,
           out_dtype=None) -> Workload:
    gen = torch.Generator().manual_seed(seed)
    x = _cast(_normal(gen, (M, K)), dtype)
    w = _cast(_normal(gen, (N, K), w_std), dtype)
    b = None
    if bias == "scalar":
        b = torch.rand(1, generator=gen, dtype=torch.float32) * 0.2 - 0.1
    od = out_dtype or ("bf16" if dtype == torch.bfloat16 else "f32")
    return Workload(name, "linear", x, w, mean_abs(x), mean_abs(w), b, od)


def conv(name, B, C, H, W, O, k, stride, padding, dilation, *, dtype=torch.float32, bias="none",
         seed=0, out_dtype=None) -> Workload:
    gen = torch.Generator().manual_seed(seed)
    x = _cast(_normal(gen, (B, C, H, W)), dtype)
    w = _cast(_normal(gen, (O, C, k, k)), dtype)
    b = None
    if bias == "channel":
        b = torch.rand(C, generator=gen, dtype=torch.float32) * 0.2 - 0.1
    elif bias == "scalar":
        b = torch.rand(1, generator=gen, dtype=torch.float32) * 0.2 - 0.1
    od = out_dtype or ("bf16" if dtype == torch.bfloat16 else "f32")
    return Workload(name, "conv", x, w, mean_abs(x), mean_abs(w), b, od, stride, padding, dilation)


# The named workloads. Seeds: 0 for the tiny linear, otherwise the workload's
# position in this list (1-based).
def tiny_linear():
    """Linear 64 x 256 x 512, fp32, no bias."""
    return linear("linear_64x256x512_f32", 64, 256, 512, seed=0)


def llm_linear():
    """Linear 4096 x 4096 x 4096, bf16, W ~ N(0, 0.02), scalar bias U(-0.1, 0.1)."""
    return linear("linear_4096x4096x4096_bf16", 4096, 4096, 4096, dtype=torch.bfloat16,
                  w_std=0.02, bias="scalar", seed=2)


def resnet_conv():
    """Conv [128,256,14,14] x [256,256,3,3], stride 1, padding 1, fp32."""
    return conv("conv_128x256x14x14_k3s1p1_f32", 128, 256, 14, 14, 256, 3, 1, 1, 1, seed=3)


def downsample_conv(dilation=1):
    """Conv [256,128,28,28] x [256,128,3,3], stride 2, bf16; padding 1 (d=1) or 2 (d=2)."""
    p = 1 if dilation == 1 else 2
    return conv(f"conv_256x128x28x28_k3s2p{p}d{dilation}_bf16", 256, 128, 28, 28, 256, 3, 2, p,
                dilation, dtype=torch.bfloat16, seed=4)


def large_linear():
    """Linear 8192 x 4096 x 11008, bf16, W ~ N(0, 0.02)."""
    return linear("linear_8192x4096x11008_bf16", 8192, 4096, 11008, dtype=torch.bfloat16,
                  w_std=0.02, seed=5)


def ragged_linear():
    """Linear 8191 x 4093 x 4100, bf16, W ~ N(0, 0.02): ragged M, N and K."""
    return linear("linear_8191x4093x4100_bf16", 8191, 4093, 4100, dtype=torch.bfloat16,
                  w_std=0.02, seed=6)


NAMED = {
    "tiny_linear": tiny_linear,
    "llm_linear": llm_linear,
    "resnet_conv": resnet_conv,
    "downsample_conv": lambda: downsample_conv(1),
    "downsample_conv_d2": lambda: downsample_conv(2),
    "large_linear": large_linear,
    "ragged_linear": ragged_linear,
}
