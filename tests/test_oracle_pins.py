"""The CPU oracle against what the definition and the mathematics fix (no GPU)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


def _torch_conv(x, w, b, stride, pad, dil, groups=1):
    # Library cross-check: torch's own CPU convolution in float64 on NCHW/KCRS views.
    xt = torch.from_numpy(x).permute(0, 3, 1, 2)
    wt = torch.from_numpy(w).permute(0, 3, 1, 2)
    bt = None if b is None else torch.from_numpy(np.asarray(b, dtype=np.float64))
    y = torch.nn.functional.conv2d(xt, wt, bt, stride=stride, padding=pad, dilation=dil, groups=groups)
    return y.permute(0, 2, 3, 1).contiguous().numpy()


@pytest.mark.parametrize("geom", [
    dict(n=2, h=9, w=8, c=8, k=12, r=3, s=3, groups=2, stride_h=1, stride_w=1, pad_h=1, pad_w=1),
    dict(n=1, h=11, w=7, c=12, k=6, r=3, s=2, groups=3, stride_h=2, stride_w=1, pad_h=1, pad_w=0, dil_w=2),
    dict(n=2, h=6, w=6, c=16, k=16, r=3, s=3, groups=16, stride_h=1, stride_w=1, pad_h=1, pad_w=1),
    dict(n=1, h=8, w=9, c=128, k=64, r=1, s=3, groups=2, stride_h=1, stride_w=2, pad_h=0, pad_w=1),
])
def test_library_grouped_conv_crosscheck(geom, oracle_lib):
    kw = dict(geom)
    wl = workloads.Workload("grp", kw.pop("n"), kw.pop("h"), kw.pop("w"), kw.pop("c"), kw.pop("k"), kw.pop("r"),
                            kw.pop("s"), bias="normal:0.1", seed=3, **kw)
    x, w, b = workloads.make_inputs(wl)
    assert w.shape == (wl.k, wl.r, wl.s, wl.c // wl.groups)
    ours = oracle.conv2d_fwd(x, w, b, **wl.options(), lib=oracle_lib)
    ref = _torch_conv(x.to(torch.float64).numpy(), w.to(torch.float64).numpy(), b.numpy(),
                      (wl.stride_h, wl.stride_w), (wl.pad_h, wl.pad_w), (wl.dil_h, wl.dil_w), wl.groups)
    assert ours.shape == ref.shape
    np.testing.assert_allclose(ours, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", range(12))
def test_library_conv_crosscheck(seed, oracle_lib):
    wl = workloads.random_small(seed, max_hw=10)
    x, w, b = workloads.make_inputs(wl)
    ours = oracle.conv2d_fwd(x, w, b, **wl.options(), lib=oracle_lib)
    xd = x.to(torch.float64).numpy()
    wd = w.to(torch.float64).numpy()
    ref = _torch_conv(xd, wd, None if b is None else b.numpy(), (wl.stride_h, wl.stride_w),
                      (wl.pad_h, wl.pad_w), (wl.dil_h, wl.dil_w))
    assert ours.shape == ref.shape
    np.testing.assert_allclose(ours, ref, rtol=1e-12, atol=1e-12)


def test_tiny_workload_matches_bruteforce(oracle_lib):
    # The parity-only tiny workload, computed two independent ways.
    wl = workloads.get("tiny_8x8_c16")
    x, w, b = workloads.make_inputs(wl)
    ours = oracle.conv2d_fwd(x, w, b, **wl.options(), lib=oracle_lib)
    brute = pins.im2col_gemm(x.to(torch.float64).numpy(), w.to(torch.float64).numpy(), b.numpy(),
                             (1, 1), (1, 1), (1, 1))
    np.testing.assert_allclose(ours, brute, rtol=1e-13, atol=1e-13)


def test_inputs_are_seeded_and_rounded():
    wl = workloads.get("resnet_56x56_c64")
    x1, w1, b1 = workloads.make_inputs(wl)
    x2, w2, b2 = workloads.make_inputs(wl)
    assert torch.equal(x1.view(torch.int16), x2.view(torch.int16))
    assert torch.equal(w1.view(torch.int16), w2.view(torch.int16))
    assert x1.dtype == torch.bfloat16 and w1.dtype == torch.bfloat16 and b1.dtype == torch.float32
    assert torch.count_nonzero(b1) == 0  # "fp32 bias zero"
    # He init: variance 2/(C*R*S) = 2/576
    var = w1.to(torch.float64).var().item()
    assert abs(var - 2 / 576) < 0.1 * 2 / 576
