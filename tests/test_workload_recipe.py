"""The synthetic inputs follow the benchmark list's recipe (CPU only): the seven workloads'
shapes and options, and the distributions their values are drawn from."""
import math

import pytest
import torch

import workloads

# (N, H, W, C, K, R, S, stride, pad, dil, x, w, bias) as the benchmark list states them.
RECIPE = {
    "tiny_8x8_c16": (1, 8, 8, 16, 16, 3, 3, 1, 1, 1, "uniform", "uniform", "uniform"),
    "resnet_56x56_c64": (4, 56, 56, 64, 64, 3, 3, 1, 1, 1, "normal", "he", "zero"),
    "resnet_28x28_c256": (16, 28, 28, 256, 256, 3, 3, 1, 1, 1, "normal", "he", "normal:0.1"),
    "splitk_7x7_c2048": (16, 7, 7, 2048, 512, 3, 3, 1, 1, 1, "uniform", "uniform", None),
    "stem_224_c3_7x7s2": (32, 224, 224, 3, 64, 7, 7, 2, 3, 1, "normal", "he", None),
    "proj_56_c256_1x1s2": (32, 56, 56, 256, 512, 1, 1, 2, 0, 1, "normal", "he", None),
    "dil2_64_c128": (8, 64, 64, 128, 128, 3, 3, 1, 2, 2, "normal", "he", None),
}


@pytest.mark.parametrize("name", sorted(RECIPE))
def test_workload_matches_the_list(name):
    n, h, w, c, k, r, s, st, pd, dl, xd, wd, bd = RECIPE[name]
    wl = workloads.get(name)
    assert (wl.n, wl.h, wl.w, wl.c, wl.k, wl.r, wl.s) == (n, h, w, c, k, r, s)
    assert (wl.stride_h, wl.stride_w, wl.pad_h, wl.pad_w, wl.dil_h, wl.dil_w) == (st, st, pd, pd, dl, dl)
    assert (wl.x_dist, wl.w_dist, wl.bias, wl.groups, wl.seed) == (xd, wd, bd, 1, 0)
    assert name in workloads.ORDER


@pytest.mark.parametrize("name", ["resnet_56x56_c64", "resnet_28x28_c256", "splitk_7x7_c2048", "tiny_8x8_c16"])
def test_value_distributions(name):
    wl = workloads.get(name)
    x, w, b = workloads.make_inputs(wl)
    assert x.dtype == torch.bfloat16 and w.dtype == torch.bfloat16 and tuple(x.shape) == (wl.n, wl.h, wl.w, wl.c)
    xf, wf = x.float(), w.float()
    if wl.x_dist == "normal":
        assert abs(float(xf.mean())) < 0.02 and abs(float(xf.var()) - 1.0) < 0.02
    else:  # uniform [-1, 1) in fp32, variance 1/3; rounding to bf16 can reach 1.0 itself
        assert float(xf.min()) >= -1.0 and float(xf.max()) <= 1.0 and abs(float(xf.var()) - 1 / 3) < 0.05
    if wl.w_dist == "he":
        assert abs(float(wf.var()) / (2.0 / (wl.c * wl.r * wl.s)) - 1.0) < 0.1
    if wl.bias == "zero":
        assert b is not None and b.dtype == torch.float32 and int(torch.count_nonzero(b)) == 0
    elif wl.bias == "normal:0.1":
        assert b.dtype == torch.float32 and abs(float(b.var()) / 0.1 - 1.0) < 0.5
    elif wl.bias is None:
        assert b is None
    # bf16 values: each is the round-to-nearest-even of an fp32 draw, so it is exactly representable
    assert torch.equal(x, x.float().to(torch.bfloat16))
    assert workloads.make_inputs(wl)[0].equal(x)  # seeded: the same every time
