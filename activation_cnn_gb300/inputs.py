"""Seeded synthetic inputs shared by the CUDA path's tests/benchmarks and the oracle.

This module only draws random numbers; it holds none of the layer's
arithmetic.  Every tensor is drawn on the CPU with its own
``torch.Generator`` whose seed is a stable function of (workload seed, tensor
name), so two independently written layer lists draw identical parameters for
a layer of the same name and shape, whatever order they enumerate layers in.

Distributions follow the workloads: conv weights He-normal
N(0, sqrt(2 / (kh*kw*C_in))) (BN folded into the bias), bias U(-0.1, 0.1),
PReLU alpha U(0, 0.25), activations U(-1, 1), U(0, 1) or N(0, 1), RGBA8
frames uniform bytes.  Values are drawn in fp32 and then cast to the storage
type (round-to-nearest-even, torch's cast), so both sides receive the same
stored values.
"""
from __future__ import annotations

import zlib

import torch

F32, F16, BF16 = 0, 1, 2
TORCH_DTYPE = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}
NHWC, NCHW = 0, 1


def _gen(seed: int, name: str) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed((int(seed) * 1_000_003 + zlib.crc32(name.encode())) % (2**63 - 1))
    return g


def tensor(seed: int, name: str, shape, dist: str = "uniform", lo: float = -1.0,
           hi: float = 1.0, std: float = 1.0, dtype: int = F32) -> torch.Tensor:
    """A CPU tensor of `shape` drawn from `dist` ('uniform' U(lo,hi) or 'normal' N(0,std))."""
    g = _gen(seed, name)
    if dist == "uniform":
        t = torch.rand(tuple(shape), generator=g, dtype=torch.float32) * (hi - lo) + lo
    elif dist == "normal":
        t = torch.randn(tuple(shape), generator=g, dtype=torch.float32) * std
    elif dist == "int":
        t = torch.randint(int(lo), int(hi) + 1, tuple(shape), generator=g).to(torch.float32)
    else:
        raise ValueError(dist)
    return t.to(TORCH_DTYPE[dtype]).contiguous()


def conv_weight(seed: int, name: str, c_out: int, c_in: int, kh: int, kw: int,
                layout: int = NHWC, dtype: int = F32) -> torch.Tensor:
    """He-normal conv weight: OHWI for NHWC activations, OIHW for NCHW."""
    std = (2.0 / (kh * kw * c_in)) ** 0.5
    shape = (c_out, kh, kw, c_in) if layout == NHWC else (c_out, c_in, kh, kw)
    return tensor(seed, name + ".w", shape, "normal", std=std, dtype=dtype)


def conv_bias(seed: int, name: str, c_out: int) -> torch.Tensor:
    return tensor(seed, name + ".b", (c_out,), "uniform", -0.1, 0.1)


def prelu_alpha(seed: int, name: str, c_out: int) -> torch.Tensor:
    return tensor(seed, name + ".alpha", (c_out,), "uniform", 0.0, 0.25)


def deconv_weight(seed: int, name: str, c_in: int, c_out: int, k: int) -> torch.Tensor:
    """Transposed-conv weight [CI, CO, K, K], fp32, He-normal over CI*K*K/4 live taps."""
    std = (2.0 / (c_in * k * k / 4.0)) ** 0.5
    return tensor(seed, name + ".w", (c_in, c_out, k, k), "normal", std=std)


def film_mlp(seed: int, name: str, c: int, hn: int):
    """Timestep MLP Linear(1, hn) -> ReLU -> Linear(hn, 2c), fp32: (w0 [hn], b0 [hn],
    w2 [2c, hn], b2 [2c]); t in [0, 1], w0 U(-2, 2), b0 U(-0.5, 0.5), w2 N(0, 0.2 / sqrt(hn))
    and b2 U(-0.05, 0.05), so the modulation 1 + s stays near 1."""
    w0 = tensor(seed, name + ".0.w", (hn,), "uniform", -2.0, 2.0)
    b0 = tensor(seed, name + ".0.b", (hn,), "uniform", -0.5, 0.5)
    w2 = tensor(seed, name + ".2.w", (2 * c, hn), "normal", std=0.2 / hn ** 0.5)
    b2 = tensor(seed, name + ".2.b", (2 * c,), "uniform", -0.05, 0.05)
    return w0, b0, w2, b2


def refine_out_weight(seed: int, name: str, c_in: int) -> torch.Tensor:
    """The refine head's last conv, [3, c_in, 3, 3] fp32, N(0, 0.25 / sqrt(9 c_in)):
    a small correction, so 2 sigmoid - 1 stays well inside (-1, 1)."""
    return tensor(seed, name + ".w", (3, c_in, 3, 3), "normal", std=0.25 / (9 * c_in) ** 0.5)


def rgba_frame(seed: int, name: str, h: int, w: int) -> torch.Tensor:
    """An [H, W, 4] uint8 frame of uniform random bytes."""
    g = _gen(seed, name)
    return torch.randint(0, 256, (h, w, 4), generator=g, dtype=torch.int32).to(torch.uint8)


def activation_shape(layout: int, n: int, c: int, h: int, w: int):
    return (n, h, w, c) if layout == NHWC else (n, c, h, w)
