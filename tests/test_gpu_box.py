"""The TMA box loader (tiles that are rectangles of output pixels, two channel chunks per
box) against the CPU oracle, element by element, through the C ABI (needs a GB300)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import check_close, gpu_conv, make_algo

pytestmark = pytest.mark.gpu

WAIT = 200_000_000  # 0.2 s bound on every device-side wait in these tests
BOX = 6


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import split_gemm_gb300
    split_gemm_gb300.load_library()
    torch.cuda.set_device(0)
    return split_gemm_gb300


def _case(n, h, w, c, k, r, s, stride=1, pad=0, dil=1, bias=True, seed=0, dist="normal"):
    def pair(v):
        return v if isinstance(v, tuple) else (v, v)
    (sh, sw), (ph, pw), (dh, dw) = pair(stride), pair(pad), pair(dil)
    wl = workloads.Workload(f"box{seed}", n, h, w, c, k, r, s, sh, sw, ph, pw, dh, dw,
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
def test_rows_rectangle_each_width(sg, bn):
    # P = Q = 12: 128-pixel tiles are 6 whole rows (72 pixels), two row blocks per image;
    # K = 200 is ragged in every tile width.
    wl, x, w, b = _case(2, 12, 12, 128, 200, 3, 3, pad=1, seed=11)
    _check(sg, wl, x, w, b, make_algo(sg, block_n=bn, loader=BOX, wait_limit_ns=WAIT), f"box bn={bn}")


@pytest.mark.parametrize("bn", [64, 128])
def test_256_pixel_rectangles(sg, bn):
    # P = Q = 22: 256-pixel tiles are 8 rows (176 pixels); the third row block is ragged.
    wl, x, w, b = _case(2, 22, 22, 256, 96, 3, 3, pad=1, seed=12)
    _check(sg, wl, x, w, b, make_algo(sg, block_m=256, block_n=bn, loader=BOX, wait_limit_ns=WAIT),
           f"box BM=256 bn={bn}")


@pytest.mark.parametrize("geom", [
    dict(n=2, h=16, w=16, c=128, k=128, r=3, s=3, pad=2, dil=2),              # dilation 2
    dict(n=2, h=15, w=15, c=128, k=64, r=3, s=3, stride=2, pad=1),            # stride 2: 8x8 outputs, 2 images per box
    dict(n=3, h=8, w=8, c=128, k=72, r=3, s=3, pad=1),                        # 2 images per box, ragged image count
    dict(n=2, h=16, w=16, c=256, k=128, r=1, s=1, stride=2),                  # 1x1 stride 2 projection
    dict(n=1, h=3, w=300, c=128, k=64, r=1, s=3, pad=(0, 1)),                 # Q > 128: part of a row per tile
    dict(n=3, h=13, w=10, c=128, k=48, r=3, s=2, stride=(2, 1), pad=(1, 0), dil=(1, 2)),  # asymmetric window
    dict(n=3, h=8, w=8, c=384, k=64, r=5, s=5, pad=2),                        # three chunk pairs per tap, 5x5
])
def test_box_geometries(sg, geom):
    kw = dict(geom)
    wl, x, w, b = _case(kw.pop("n"), kw.pop("h"), kw.pop("w"), kw.pop("c"), kw.pop("k"), kw.pop("r"), kw.pop("s"),
                        seed=13, **kw)
    _check(sg, wl, x, w, b, make_algo(sg, loader=BOX, wait_limit_ns=WAIT), wl.describe())


@pytest.mark.parametrize("bm", [128, 256])
def test_box_pixel_count_not_a_multiple_of_8(sg, bm):
    # 7 x 7 images: boxes of 2 (bm 128) or 5 (bm 256) whole images hold 98 or 245 pixels, so the
    # second channel chunk of every box starts mid-way through a 1024-byte swizzle atom.
    wl, x, w, b = _case(6, 7, 7, 256, 128, 3, 3, pad=1, seed=20)
    _check(sg, wl, x, w, b, make_algo(sg, loader=BOX, block_m=bm, block_n=128, wait_limit_ns=WAIT),
           f"box 7x7 BM={bm}")


@pytest.mark.parametrize("reduction", [1, 2])
@pytest.mark.parametrize("splits", [2, 3])
def test_box_split_k(sg, splits, reduction):
    wl, x, w, b = _case(2, 12, 12, 256, 96, 3, 3, pad=1, seed=14)
    algo = make_algo(sg, loader=BOX, splits=splits, wait_limit_ns=WAIT, reduction=reduction)
    got = _check(sg, wl, x, w, b, algo, f"box splits={splits} reduction={reduction}")
    if reduction == 1:  # the ordered reduction is bitwise reproducible
        assert np.array_equal(got, gpu_conv(sg, x, w, b, wl.options(), algo=algo))


@pytest.mark.parametrize("grid", [1, 5, 7])
def test_box_stream_k(sg, grid):
    # 4 tiles x 9 stages; grid 5 and 7 cut tiles between CTAs, grid 1 runs them all on one CTA.
    wl, x, w, b = _case(2, 12, 12, 256, 256, 3, 3, pad=1, seed=15)
    _check(sg, wl, x, w, b, make_algo(sg, loader=BOX, grid=grid, wait_limit_ns=WAIT), f"box grid={grid}")


def test_box_integer_inputs_exact(sg):
    # Small integers: every partial sum is exact in fp32, so the GPU result equals the oracle's.
    wl, x, w, b = _case(2, 12, 12, 128, 64, 3, 3, pad=1, seed=16, dist="int:-3:3")
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=BOX, wait_limit_ns=WAIT))
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    assert np.array_equal(got.astype(np.float64), ref)


def test_box_matches_im2col_loader(sg):
    # The two TMA loaders sum the same products; they agree within the tolerance.
    wl, x, w, b = _case(4, 14, 14, 256, 128, 3, 3, pad=1, seed=17)
    box = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=BOX, wait_limit_ns=WAIT))
    im2col = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=1, wait_limit_ns=WAIT))
    check_close(box, im2col.astype(np.float64), wl.c, wl.r, wl.s, "box vs im2col")


def test_box_rejects_unsupported(sg):
    import split_gemm_gb300 as m
    # C = 64: two chunks per box need C % 128 == 0.
    wl, x, w, b = _case(1, 8, 8, 64, 64, 3, 3, pad=1, seed=18)
    with pytest.raises(m.Conv2dError):
        gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=BOX))
    # 256-pixel box tiles hold at most 128 output channels.
    wl, x, w, b = _case(1, 16, 16, 128, 256, 3, 3, pad=1, seed=19)
    with pytest.raises(m.Conv2dError):
        gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=BOX, block_m=256, block_n=256))
