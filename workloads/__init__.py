"""Seeded synthetic inputs for the 2-D convolution forward workloads.

This module is shared by the CPU oracle side (``oracle/``) and the CUDA side
(``split_gemm_gb300``) and holds none of the convolution's arithmetic: it only
names each workload's shapes and options and draws its inputs.  Output extents,
FLOP counts and everything else that depends on the convolution definition live
with each side separately.

Value recipe (one ``torch.Generator('cpu')`` per workload, seeded, drawn in this
order: input, then weight, then bias):

* every value is drawn in fp32 and then rounded to bfloat16 with
  round-to-nearest-even (``Tensor.to(torch.bfloat16)``); those bf16 values are
  the inputs of both sides;
* ``uniform``  -> U[-1, 1);
* ``normal``   -> N(0, 1);
* ``he``       -> N(0, 2 / (C*R*S)), i.e. variance 2/fan_in (He init);
* the bias stays fp32 (it is never rounded);
* ``N(0, v)`` in a workload description means variance ``v``.

Layouts: input NHWC, weight KRSC (output channel, filter row, filter column,
input channel), bias [K], all contiguous.  These are the layouts that burn's
``conv_forward`` produces before its implicit-GEMM kernel runs (docs.rs
burn-cubecl 0.20.0, ``burn_cubecl/kernel/conv/base.rs``, ``conv_forward``: both
input and weight go through ``permute_nchw_to_nhwc``).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

__all__ = ["Workload", "WORKLOADS", "get", "make_inputs", "make_output_grad", "random_small"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n: int
    h: int
    w: int
    c: int
    k: int
    r: int
    s: int
    stride_h: int = 1
    stride_w: int = 1
    pad_h: int = 0
    pad_w: int = 0
    dil_h: int = 1
    dil_w: int = 1
    x_dist: str = "normal"      # "uniform" | "normal" | "int:<lo>:<hi>"
    w_dist: str = "he"          # "uniform" | "normal" | "he" | "int:<lo>:<hi>"
    bias: Optional[str] = None  # None | "zero" | "uniform" | "normal:<variance>" | "int:<lo>:<hi>"
    seed: int = 0
    note: str = ""
    groups: int = 1  # channels split into consecutive groups; weight [K][R][S][C/groups]

    def options(self) -> dict:
        return dict(stride=(self.stride_h, self.stride_w), padding=(self.pad_h, self.pad_w),
                    dilation=(self.dil_h, self.dil_w), groups=self.groups)

    def describe(self) -> str:
        return (f"N{self.n} H{self.h} W{self.w} C{self.c} K{self.k} {self.r}x{self.s} "
                f"s{self.stride_h}x{self.stride_w} p{self.pad_h}x{self.pad_w} d{self.dil_h}x{self.dil_w}"
                + (f" g{self.groups}" if self.groups != 1 else ""))


# The seven workloads of the build's benchmark list.  Shapes and distributions
# follow the benchmark description; the pages themselves print no conv shape
# (burn PR #2287, "Benchmarking / Conv2d": medians only).
WORKLOADS = {
    wl.name: wl for wl in [
        Workload("tiny_8x8_c16", 1, 8, 8, 16, 16, 3, 3, 1, 1, 1, 1, 1, 1,
                 x_dist="uniform", w_dist="uniform", bias="uniform",
                 note="parity-only tiny case (GEMM 64x16x144)"),
        Workload("resnet_56x56_c64", 4, 56, 56, 64, 64, 3, 3, 1, 1, 1, 1, 1, 1,
                 x_dist="normal", w_dist="he", bias="zero",
                 note="GEMM 12544x64x576, fp32 zero bias buffer"),
        Workload("resnet_28x28_c256", 16, 28, 28, 256, 256, 3, 3, 1, 1, 1, 1, 1, 1,
                 x_dist="normal", w_dist="he", bias="normal:0.1",
                 note="GEMM 12544x256x2304"),
        Workload("splitk_7x7_c2048", 16, 7, 7, 2048, 512, 3, 3, 1, 1, 1, 1, 1, 1,
                 x_dist="uniform", w_dist="uniform", bias=None,
                 note="small M*N, long reduction: GEMM 784x512x18432"),
        Workload("stem_224_c3_7x7s2", 32, 224, 224, 3, 64, 7, 7, 2, 2, 3, 3, 1, 1,
                 x_dist="normal", w_dist="he", bias=None,
                 note="C*R*S=147, not a multiple of 16: GEMM 401408x64x147"),
        Workload("proj_56_c256_1x1s2", 32, 56, 56, 256, 512, 1, 1, 2, 2, 0, 0, 1, 1,
                 x_dist="normal", w_dist="he", bias=None,
                 note="strided 1x1 projection: GEMM 25088x512x256"),
        Workload("dil2_64_c128", 8, 64, 64, 128, 128, 3, 3, 1, 1, 2, 2, 2, 2,
                 x_dist="normal", w_dist="he", bias=None,
                 note="dilation 2: GEMM 32768x128x1152"),
    ]
}

# Grouped convolutions (beyond the benchmark list): a ResNeXt-style 3x3 layer with
# 32 groups of 8 channels, one with 8 groups of 64 channels, and a depthwise 3x3.
GROUPED = {
    wl.name: wl for wl in [
        Workload("resnext_28x28_c256_g32", 16, 28, 28, 256, 256, 3, 3, 1, 1, 1, 1, 1, 1,
                 x_dist="normal", w_dist="he", bias="normal:0.1", groups=32,
                 note="32 groups of 8 channels: 32 GEMMs 12544x8x72"),
        Workload("grouped_28x28_c512_g8", 16, 28, 28, 512, 512, 3, 3, 1, 1, 1, 1, 1, 1,
                 x_dist="normal", w_dist="he", bias="normal:0.1", groups=8,
                 note="8 groups of 64 channels: 8 GEMMs 12544x64x576"),
        Workload("depthwise_56x56_c128", 16, 56, 56, 128, 128, 3, 3, 1, 1, 1, 1, 1, 1,
                 x_dist="normal", w_dist="he", bias="normal:0.1", groups=128,
                 note="depthwise 3x3 (one channel per group), MobileNet-style"),
    ]
}
WORKLOADS.update(GROUPED)

# Order in which the benchmark list names them.
ORDER = ["tiny_8x8_c16", "resnet_56x56_c64", "resnet_28x28_c256", "splitk_7x7_c2048",
         "stem_224_c3_7x7s2", "proj_56_c256_1x1s2", "dil2_64_c128"]


def get(name: str) -> Workload:
    return WORKLOADS[name]


def _draw(gen: torch.Generator, shape, dist: str, fan_in: int) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    if dist == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32)
    if dist == "he":
        return torch.randn(shape, generator=gen, dtype=torch.float32) * math.sqrt(2.0 / fan_in)
    if dist.startswith("normal:"):
        var = float(dist.split(":")[1])
        return torch.randn(shape, generator=gen, dtype=torch.float32) * math.sqrt(var)
    if dist.startswith("int:"):
        _, lo, hi = dist.split(":")
        return torch.randint(int(lo), int(hi) + 1, shape, generator=gen).to(torch.float32)
    if dist == "zero":
        return torch.zeros(shape, dtype=torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def make_inputs(wl: Workload, seed: Optional[int] = None):
    """Return (x, w, bias) on the CPU: x [N,H,W,C] bf16, w [K,R,S,C/groups] bf16, bias [K] fp32 or None."""
    gen = torch.Generator("cpu")
    gen.manual_seed(wl.seed if seed is None else seed)
    cg = wl.c // wl.groups
    fan_in = cg * wl.r * wl.s
    x = _draw(gen, (wl.n, wl.h, wl.w, wl.c), wl.x_dist, fan_in).to(torch.bfloat16).contiguous()
    w = _draw(gen, (wl.k, wl.r, wl.s, cg), wl.w_dist, fan_in).to(torch.bfloat16).contiguous()
    b = None
    if wl.bias is not None:
        b = _draw(gen, (wl.k,), wl.bias, fan_in).contiguous()
    return x, w, b


def output_extent(in_size: int, pad: int, dil: int, ker: int, stride: int) -> int:
    """Output size along one axis (the shape of the output gradient only; no arithmetic of the method)."""
    room = in_size + 2 * pad - (dil * (ker - 1) + 1)
    return 0 if room < 0 else room // stride + 1


def make_output_grad(wl: Workload, seed: Optional[int] = None, variance: Optional[float] = None) -> torch.Tensor:
    """An output gradient dy [N,P,Q,K] bf16 for a workload's backward passes, drawn in fp32
    from its own generator (seed + 7919) and rounded to bf16.

    Default variance 2/L with L = N*P*Q, the reduction length of every weight-gradient
    element (the He scaling the forward weights use for theirs); the data gradient, whose
    reduction runs over K*R*S against the He-init weights, takes ``variance=1.0``."""
    p = output_extent(wl.h, wl.pad_h, wl.dil_h, wl.r, wl.stride_h)
    q = output_extent(wl.w, wl.pad_w, wl.dil_w, wl.s, wl.stride_w)
    gen = torch.Generator("cpu")
    gen.manual_seed((wl.seed if seed is None else seed) + 7919)
    var = 2.0 / max(1, wl.n * p * q) if variance is None else float(variance)
    return (torch.randn((wl.n, p, q, wl.k), generator=gen, dtype=torch.float32) * math.sqrt(var)).to(
        torch.bfloat16).contiguous()


def random_small(seed: int, *, max_hw: int = 12, channels=(1, 3, 8, 16, 24, 64),
                 ints: bool = False) -> Workload:
    """A random small workload for sweeps (shapes only depend on ``seed``).

    Draws stride, padding, dilation and filter size independently per axis so
    that asymmetric cases occur; rejects draws whose window does not fit.
    """
    g = torch.Generator("cpu")
    g.manual_seed(10_000 + seed)

    def pick(seq):
        return seq[int(torch.randint(0, len(seq), (1,), generator=g))]

    while True:
        n = pick([1, 2, 3])
        h = pick(list(range(1, max_hw + 1)))
        w_ = pick(list(range(1, max_hw + 1)))
        c = pick(list(channels))
        k = pick([1, 5, 16, 32, 48, 64, 80, 130])
        r = pick([1, 2, 3, 5])
        s = pick([1, 2, 3, 5])
        sh, sw = pick([1, 2, 3]), pick([1, 2, 3])
        ph, pw = pick([0, 1, 2, 3]), pick([0, 1, 2, 3])
        dh, dw = pick([1, 2, 3]), pick([1, 2, 3])
        if h + 2 * ph >= dh * (r - 1) + 1 and w_ + 2 * pw >= dw * (s - 1) + 1:
            break
    dist = "int:-3:3" if ints else None
    return Workload(f"rand{seed}", n, h, w_, c, k, r, s, sh, sw, ph, pw, dh, dw,
                    x_dist=dist or "normal", w_dist=dist or "he",
                    bias=(dist or "normal:0.1") if seed % 2 == 0 else None, seed=seed)
