"""Fused-epilogue steps of the CPU reference -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use this module.  It shares no code with the CUDA path.

The fused epilogue takes the convolution's exact value u = conv(x, w) + bias
(the fp64 output of the direct convolution) through two optional steps, in
this order:

1. activation: ReLU, max(u, 0);
2. output type: bf16, the value rounded to the nearest bfloat16 (ties to the
   even significand), the same rounding the workloads use to make their bf16
   inputs.

The half-precision output at the end of the epilogue is the case NVIDIA/Fuser
issue #1316 ("Split-K matmul is slow even for few partitions", the comment on
aliasing the output as the reduction work buffer) names as the common one; the
activation step is the plain reading of "fused activation" (elementwise, after
the bias).  ``round_bf16`` is written from the definition of the format: 8
significant bits, exponent range of IEEE binary32, subnormals below 2**-126.

Pinned by ``tests/test_oracle_epilogue.py`` (every bf16 value is a fixed point,
midpoints go to the even neighbour, a library fp32->bf16 cast agrees on random
and subnormal inputs, overflow to infinity, a hand-worked ReLU-after-bias case)
and its mutation tests.
"""
from __future__ import annotations

from typing import Optional, Tuple

import numpy as np

BF16_SIG_BITS = 8             # significant bits including the implicit one
BF16_MIN_NORMAL_EXP = -126    # smallest normal binade 2**-126 (same as binary32)
BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def relu(u: np.ndarray) -> np.ndarray:
    """max(u, 0) elementwise."""
    return np.maximum(np.asarray(u, dtype=np.float64), 0.0)


def round_bf16(v: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to even; returns float64.

    For |v| in [2**e, 2**(e+1)) the spacing of bf16 values is 2**(e - 7); below
    the normal range it stays 2**(-126 - 7).  v / spacing is an exact fp64
    number; rounding it to the nearest integer with ties to even (np.rint)
    rounds the significand.  A result above the largest finite bf16 value is
    an overflow to infinity.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros_like(v)
    finite = np.isfinite(v) & (v != 0.0)
    a = v[finite]
    _, e1 = np.frexp(np.abs(a))          # |a| = m * 2**e1, 0.5 <= m < 1, so |a| in [2**(e1-1), 2**e1)
    e = np.maximum(e1 - 1, BF16_MIN_NORMAL_EXP)
    spacing = np.ldexp(1.0, e - (BF16_SIG_BITS - 1))
    r = np.rint(a / spacing) * spacing
    r = np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, r), r)
    out[finite] = r
    out[~finite] = v[~finite]            # zeros, infinities and NaNs pass through
    return out


def apply(u: np.ndarray, relu_on: bool, out_bf16: bool) -> np.ndarray:
    """The fused epilogue on the exact values u: activation, then the output rounding."""
    y = relu(u) if relu_on else np.asarray(u, dtype=np.float64)
    return round_bf16(y) if out_bf16 else y


def bracket(u: np.ndarray, bound: np.ndarray, relu_on: bool, out_bf16: bool) -> Tuple[np.ndarray, np.ndarray]:
    """Range [lo, hi] that an epilogue output may take when its pre-epilogue fp32 value f
    satisfies |f - u| <= bound.

    Both steps are monotone, so the output of any such f lies between the
    outputs of u - bound and u + bound.  With a bf16 output, where lo == hi the
    stored value is determined exactly.
    """
    u = np.asarray(u, dtype=np.float64)
    bound = np.asarray(bound, dtype=np.float64)
    return apply(u - bound, relu_on, out_bf16), apply(u + bound, relu_on, out_bf16)


def conv2d_fwd_fused(x, w, bias=None, stride=1, padding=0, dilation=1, groups=1, *, relu_on: bool = False,
                     out_bf16: bool = False, threads: Optional[int] = None) -> Tuple[np.ndarray, np.ndarray]:
    """(u, y): the exact convolution with bias u (float64, NHWC) and the fused epilogue's output y."""
    from . import conv2d_fwd
    u = conv2d_fwd(x, w, bias, stride, padding, dilation, threads=threads, groups=groups)
    return u, apply(u, relu_on, out_bf16)
