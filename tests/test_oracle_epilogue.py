"""Pins for the oracle's fused-epilogue steps (ReLU, bf16 output rounding), and
mutants of those steps that the pins must reject.

The rounding is pinned to the format's definition (every bf16 value is a fixed
point, midpoints go to the even neighbour, overflow goes to infinity) and to a
library cast (torch's fp32 -> bf16 conversion, round to nearest even) on
random, subnormal and large fp32 values, where rounding once from fp64 and
once from fp32 agree because the inputs are fp32 values.  The activation is
pinned by a hand-worked case in which ReLU must act after the bias.
"""
from __future__ import annotations

import os
import types

import numpy as np
import pytest
import torch

from oracle import epilogue

_SRC = os.path.join(os.path.dirname(epilogue.__file__), "epilogue.py")


def _all_finite_bf16() -> np.ndarray:
    bits = np.arange(1 << 16, dtype=np.uint32)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # drop infinities and NaNs (exponent all ones)
    return (bits << 16).view(np.float32).astype(np.float64)


def _positive_finite_bf16_sorted() -> np.ndarray:
    bits = np.arange(0, 0x7F80, dtype=np.uint32)  # +0 .. largest finite
    return (bits << 16).view(np.float32).astype(np.float64)


def _torch_bf16(v32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(v32.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


# ---------------------------------------------------------------- the pins

def pin_fixed_points(mod) -> None:
    vals = _all_finite_bf16()
    got = mod.round_bf16(vals)
    assert np.array_equal(got, vals), "a bf16 value is not a fixed point of the rounding"


def pin_midpoints_to_even(mod) -> None:
    vals = _positive_finite_bf16_sorted()
    lo, hi = vals[:-1], vals[1:]
    mid = (lo + hi) / 2.0                      # exact in fp64
    lo_bits = np.arange(0, 0x7F80 - 1, dtype=np.uint32)
    even = np.where(lo_bits % 2 == 0, lo, hi)  # the neighbour whose significand is even
    got = mod.round_bf16(mid)
    assert np.array_equal(got, even), "a midpoint did not round to the even neighbour"
    assert np.array_equal(mod.round_bf16(-mid), -even), "rounding is not symmetric in sign"
    below = np.nextafter(mid, -np.inf)
    above = np.nextafter(mid, np.inf)
    assert np.array_equal(mod.round_bf16(below), lo), "a value just below a midpoint did not round down"
    assert np.array_equal(mod.round_bf16(above), hi), "a value just above a midpoint did not round up"


def pin_library_cast(mod) -> None:
    rng = np.random.default_rng(7)
    parts = [
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(5000) * 1e30).astype(np.float32),
        (rng.uniform(-1, 1, 5000) * 2.0 ** -130).astype(np.float32),   # subnormal in binary32
        (rng.uniform(-1, 1, 5000) * 2.0 ** -120).astype(np.float32),
        np.array([3.3895314e38, -3.3895314e38, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8], dtype=np.float32),
    ]
    v32 = np.concatenate(parts)
    got = mod.round_bf16(v32.astype(np.float64))
    want = _torch_bf16(v32)
    assert np.array_equal(got, want), "rounding disagrees with the library fp32 -> bf16 cast"


def pin_overflow(mod) -> None:
    mx = epilogue.BF16_MAX
    half = 2.0 ** 119                      # half the spacing in the top binade
    assert mod.round_bf16(np.array([mx + half]))[0] == np.inf       # tie: the even neighbour is 2**128
    assert mod.round_bf16(np.array([mx + half * 0.99]))[0] == mx
    assert mod.round_bf16(np.array([-(mx + half)]))[0] == -np.inf
    assert mod.round_bf16(np.array([0.0]))[0] == 0.0


def pin_relu_after_bias(mod) -> None:
    # 1x1 convolutions of one pixel: acc = x*w, u = acc + bias.
    x = np.array([[[[1.0]]], [[[1.0]]], [[[-2.0]]]])
    w = np.array([[[[2.0]]]])
    bias = np.array([-3.0])
    acc = x.reshape(-1) * w.reshape(-1)               # 2, 2, -4
    u = acc + bias                                    # -1, -1, -7
    got = mod.apply(u, True, False)
    assert np.array_equal(got, np.array([0.0, 0.0, 0.0]))
    u2 = acc + 3.0                                    # 5, 5, -1
    assert np.array_equal(mod.apply(u2, True, False), np.array([5.0, 5.0, 0.0]))
    assert np.array_equal(mod.apply(u2, False, False), u2)
    # bf16 output of values that need rounding: 1 + 2**-8 is a tie (-> 1), 1 + 3*2**-8 -> 1 + 2**-6.
    got = mod.apply(np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8]), True, True)
    assert np.array_equal(got, np.array([1.0, 1.0 + 2 ** -6, 0.0]))


def pin_fused_conv(mod) -> None:
    """The oracle's fused call equals a library convolution's output put through ReLU and the cast."""
    g = torch.Generator().manual_seed(3)
    x = torch.randn(2, 6, 7, 16, generator=g).to(torch.bfloat16)
    w = torch.randn(8, 3, 3, 16, generator=g).to(torch.bfloat16)
    b = torch.randn(8, generator=g)
    u, y = epilogue.conv2d_fwd_fused(x, w, b, 1, 1, 1, relu_on=True, out_bf16=False, threads=2)
    ref = torch.nn.functional.conv2d(x.double().permute(0, 3, 1, 2), w.double().permute(0, 3, 1, 2),
                                     b.double(), padding=1).permute(0, 2, 3, 1).numpy()
    assert np.allclose(u, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(mod.apply(u, True, False), np.maximum(ref, 0.0), rtol=1e-12, atol=1e-12)
    # Values that fp32 holds exactly: the oracle's bf16 rounding of them is the library cast.
    u32 = u.astype(np.float32)
    got = mod.apply(u32.astype(np.float64), True, True)
    want = torch.relu(torch.from_numpy(u32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(got, want)


def pin_bracket(mod) -> None:
    u = np.array([1.0 + 2 ** -9, -0.25, 1.0 + 2 ** -8])
    b = np.full(3, 2.0 ** -12)
    lo, hi = mod.bracket(u, b, True, True)
    assert np.array_equal(lo, np.array([1.0, 0.0, 1.0]))
    assert np.array_equal(hi, np.array([1.0, 0.0, 1.0 + 2 ** -7]))


ALL = [pin_fixed_points, pin_midpoints_to_even, pin_library_cast, pin_overflow, pin_relu_after_bias,
       pin_fused_conv, pin_bracket]


@pytest.mark.parametrize("pin", ALL, ids=lambda f: f.__name__)
def test_epilogue_pin(pin):
    pin(epilogue)


# ---------------------------------------------------------------- mutants

def _mutant(old: str, new: str):
    src = open(_SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
    mod = types.ModuleType("epilogue_mutant")
    mod.__dict__["__name__"] = "oracle.epilogue_mutant"
    mod.__dict__["__package__"] = "oracle"
    exec(compile(src.replace(old, new), _SRC + " (mutant)", "exec"), mod.__dict__)
    return mod


MUTANTS = {
    "truncate_instead_of_round": ("np.rint(a / spacing)", "np.trunc(a / spacing)"),
    "ties_away_from_zero": ("np.rint(a / spacing)", "(np.sign(a) * np.floor(np.abs(a / spacing) + 0.5))"),
    "one_significant_bit_too_many": ("BF16_SIG_BITS = 8 ", "BF16_SIG_BITS = 9 "),
    "one_significant_bit_too_few": ("BF16_SIG_BITS = 8 ", "BF16_SIG_BITS = 7 "),
    "binade_off_by_one": ("np.maximum(e1 - 1, BF16_MIN_NORMAL_EXP)", "np.maximum(e1, BF16_MIN_NORMAL_EXP)"),
    "no_subnormal_floor": ("np.maximum(e1 - 1, BF16_MIN_NORMAL_EXP)", "(e1 - 1)"),
    "no_overflow_to_inf": ("np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, r), r)", "r"),
    "relu_as_abs": ("np.maximum(np.asarray(u, dtype=np.float64), 0.0)", "np.abs(np.asarray(u, dtype=np.float64))"),
    "relu_leaks_negatives": ("np.maximum(np.asarray(u, dtype=np.float64), 0.0)",
                             "np.where(np.asarray(u) > 0, u, 0.01 * np.asarray(u, dtype=np.float64))"),
    "rounding_skipped": ("return round_bf16(y) if out_bf16 else y", "return y"),
    "activation_skipped": ("y = relu(u) if relu_on else", "y = u if relu_on else"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_epilogue_mutant_is_caught(name):
    old, new = MUTANTS[name]
    mod = _mutant(old, new)
    failures = 0
    for pin in ALL:
        try:
            pin(mod)
        except AssertionError:
            failures += 1
    assert failures > 0, f"mutant {name} passed every pin"
