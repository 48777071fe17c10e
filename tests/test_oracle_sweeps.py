"""Seeded random-shape sweeps of the three oracles against torch's float64 convolution and
its gradients (CPU only).  The shapes come from workloads.random_small (random strides,
pads, dilations and filter sizes per axis) with a random divisor of C and K as the group
count, so every option combination the oracles accept is exercised somewhere."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import dgrad as od
from oracle import wgrad as ow

SEEDS = range(24)


def _grouped(seed):
    wl = workloads.random_small(seed)
    g = int(np.gcd(wl.c, wl.k))
    divisors = [d for d in range(1, g + 1) if g % d == 0]
    groups = divisors[seed % len(divisors)]
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((wl.n, wl.h, wl.w, wl.c))
    w = rng.standard_normal((wl.k, wl.r, wl.s, wl.c // groups))
    opts = dict(stride=(wl.stride_h, wl.stride_w), padding=(wl.pad_h, wl.pad_w), dilation=(wl.dil_h, wl.dil_w))
    return x, w, groups, opts


def _nchw(a):
    return torch.from_numpy(a).permute(0, 3, 1, 2)


@pytest.mark.parametrize("seed", SEEDS)
def test_forward_matches_library(seed):
    x, w, groups, opts = _grouped(seed)
    got = oracle.conv2d_fwd_f64(x, w, None, **opts, groups=groups, threads=2)
    ref = torch.nn.functional.conv2d(_nchw(x), _nchw(w), None, groups=groups, **opts).permute(0, 2, 3, 1).numpy()
    assert np.allclose(got, ref, rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("seed", SEEDS)
def test_gradients_match_library(seed):
    x, w, groups, opts = _grouped(seed)
    y = oracle.conv2d_fwd_f64(x, w, None, **opts, groups=groups, threads=2)
    dy = np.random.default_rng(1000 + seed).standard_normal(y.shape)
    dw = ow.conv2d_wgrad_f64(x, dy, w.shape, **opts, groups=groups, threads=2)
    dx = od.conv2d_dgrad_f64(dy, w, x.shape, **opts, groups=groups, threads=2)
    k, r, s, cg = w.shape
    ref_dw = torch.nn.grad.conv2d_weight(_nchw(x), (k, cg, r, s), _nchw(dy), groups=groups,
                                         **opts).permute(0, 2, 3, 1).numpy()
    n, h, wd, c = x.shape
    ref_dx = torch.nn.grad.conv2d_input((n, c, h, wd), _nchw(w), _nchw(dy), groups=groups,
                                        **opts).permute(0, 2, 3, 1).numpy()
    assert np.allclose(dw, ref_dw, rtol=1e-10, atol=1e-10)
    assert np.allclose(dx, ref_dx, rtol=1e-10, atol=1e-10)
