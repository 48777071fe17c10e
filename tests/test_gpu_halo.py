"""The halo loader (stride 1: tiles of 128 consecutive pixels of an image seen with
the padded row pitch, one TMA box of whole padded input rows per 64-channel chunk
serving every filter tap) against the CPU oracle, element by element, through the
C ABI (needs a GB300)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import check_close, gpu_conv, make_algo

pytestmark = pytest.mark.gpu

WAIT = 200_000_000  # 0.2 s bound on every device-side wait in these tests
HALO = 7


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import split_gemm_gb300
    split_gemm_gb300.load_library()
    torch.cuda.set_device(0)
    return split_gemm_gb300


def _case(n, h, w, c, k, r, s, pad=0, dil=1, bias=True, seed=0, dist="normal"):
    def pair(v):
        return v if isinstance(v, tuple) else (v, v)
    (ph, pw), (dh, dw) = pair(pad), pair(dil)
    wl = workloads.Workload(f"halo{seed}", n, h, w, c, k, r, s, 1, 1, ph, pw, dh, dw,
                            x_dist=dist, w_dist="he" if dist == "normal" else dist,
                            bias=("normal:0.1" if dist == "normal" else dist) if bias else None, seed=seed)
    x, wt, b = workloads.make_inputs(wl)
    return wl, x, wt, b


def _check(sg, wl, x, w, b, algo, what):
    got = gpu_conv(sg, x, w, b, wl.options(), algo=algo)
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    check_close(got, ref, wl.c, wl.r, wl.s, what)
    return got


@pytest.mark.parametrize("bn", [64, 128, 256])
def test_each_width(sg, bn):
    # 12 x 12 output, row pitch 14: 168 virtual pixels per image = 2 tiles, the second
    # ragged; K = 200 is ragged in every tile width; 2 chunks x 9 taps.
    wl, x, w, b = _case(2, 12, 12, 128, 200, 3, 3, pad=1, seed=21)
    _check(sg, wl, x, w, b, make_algo(sg, block_n=bn, loader=HALO, wait_limit_ns=WAIT), f"halo bn={bn}")


@pytest.mark.parametrize("geom", [
    dict(n=2, h=16, w=16, c=128, k=128, r=3, s=3, pad=2, dil=2),             # dilation 2
    dict(n=1, h=20, w=30, c=64, k=64, r=5, s=5, pad=2),                      # 5x5, one chunk
    dict(n=3, h=9, w=7, c=192, k=72, r=3, s=2, pad=(1, 0), dil=(2, 1)),      # asymmetric window, 3 chunks
    dict(n=2, h=10, w=10, c=64, k=64, r=3, s=3, pad=0),                      # no padding (valid convolution)
    dict(n=1, h=4, w=100, c=64, k=96, r=3, s=3, pad=1),                      # long rows: a tile is part of a row
    dict(n=2, h=17, w=5, c=64, k=64, r=1, s=3, pad=(0, 1)),                  # 1 x 3 filter
    dict(n=2, h=6, w=6, c=128, k=64, r=3, s=3, pad=3),                       # padding wider than the filter reach
])
def test_geometries(sg, geom):
    kw = dict(geom)
    wl, x, w, b = _case(kw.pop("n"), kw.pop("h"), kw.pop("w"), kw.pop("c"), kw.pop("k"), kw.pop("r"), kw.pop("s"),
                        seed=22, **kw)
    _check(sg, wl, x, w, b, make_algo(sg, loader=HALO, wait_limit_ns=WAIT), wl.describe())


@pytest.mark.parametrize("reduction", [1, 2])
@pytest.mark.parametrize("splits", [2, 5])
def test_split_k(sg, splits, reduction):
    # Splits cut chunks in the middle of their taps: each segment loads its own halo.
    wl, x, w, b = _case(2, 12, 12, 256, 96, 3, 3, pad=1, seed=23)
    algo = make_algo(sg, loader=HALO, splits=splits, wait_limit_ns=WAIT, reduction=reduction)
    got = _check(sg, wl, x, w, b, algo, f"halo splits={splits} reduction={reduction}")
    if reduction == 1:  # the ordered reduction is bitwise reproducible
        assert np.array_equal(got, gpu_conv(sg, x, w, b, wl.options(), algo=algo))


@pytest.mark.parametrize("grid", [1, 3, 7, 11])
def test_stream_k(sg, grid):
    # 4 tiles x 36 stages; grids 3, 7 and 11 cut tiles (and chunks) between CTAs, grid 1
    # runs every tile on one CTA through both halo buffers and both accumulators.
    wl, x, w, b = _case(2, 12, 12, 256, 256, 3, 3, pad=1, seed=24)
    _check(sg, wl, x, w, b, make_algo(sg, loader=HALO, grid=grid, block_n=128, wait_limit_ns=WAIT),
           f"halo grid={grid}")


def test_integer_inputs_exact(sg):
    # Small integers: every partial sum is exact in fp32, so the GPU result equals the oracle's.
    wl, x, w, b = _case(2, 12, 12, 128, 64, 3, 3, pad=1, seed=25, dist="int:-3:3")
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=HALO, wait_limit_ns=WAIT))
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    assert np.array_equal(got.astype(np.float64), ref)


def test_matches_im2col_loader(sg):
    # The halo and im2col loaders sum the same products in different orders.
    wl, x, w, b = _case(4, 14, 14, 256, 128, 3, 3, pad=1, seed=26)
    halo = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=HALO, wait_limit_ns=WAIT))
    im2col = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=1, wait_limit_ns=WAIT))
    check_close(halo, im2col.astype(np.float64), wl.c, wl.r, wl.s, "halo vs im2col")


@pytest.mark.parametrize("name", ["resnet_56x56_c64", "resnet_28x28_c256", "dil2_64_c128"])
def test_full_workload(sg, name):
    # The stride-1 benchmark shapes at full size through the halo loader.
    wl = workloads.get(name)
    x, w, b = workloads.make_inputs(wl)
    _check(sg, wl, x, w, b, make_algo(sg, loader=HALO, wait_limit_ns=WAIT), name + " halo")


def test_rejects_unsupported(sg):
    import split_gemm_gb300 as m
    # Stride 2 has no halo layout.
    wl = workloads.Workload("halo_s2", 1, 16, 16, 64, 64, 3, 3, 2, 2, 1, 1, 1, 1, seed=27)
    x, w, b = workloads.make_inputs(wl)
    with pytest.raises(m.Conv2dError):
        gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=HALO))
    # C % 64 != 0.
    wl, x, w, b = _case(1, 8, 8, 32, 64, 3, 3, pad=1, seed=28)
    with pytest.raises(m.Conv2dError):
        gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=HALO))
    # Padded rows wider than a TMA box (256 pixels).
    wl, x, w, b = _case(1, 2, 300, 64, 64, 1, 3, pad=(0, 1), seed=29)
    with pytest.raises(m.Conv2dError):
        gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=HALO))
