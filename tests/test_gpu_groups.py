"""Grouped convolution (channels split into consecutive groups, weight [K][R][S][C/groups])
against the CPU oracle, element by element, through the C ABI (needs a GB300)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import check_close, gpu_conv, make_algo

pytestmark = pytest.mark.gpu

WAIT = 200_000_000  # 0.2 s bound on every device-side wait in these tests


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import split_gemm_gb300
    split_gemm_gb300.load_library()
    torch.cuda.set_device(0)
    return split_gemm_gb300


def _case(n, h, w, c, k, r, s, groups, stride=1, pad=0, dil=1, bias=True, seed=0, dist="normal"):
    def pair(v):
        return v if isinstance(v, tuple) else (v, v)
    (sh, sw), (ph, pw), (dh, dw) = pair(stride), pair(pad), pair(dil)
    wl = workloads.Workload(f"grp{seed}", n, h, w, c, k, r, s, sh, sw, ph, pw, dh, dw,
                            x_dist=dist, w_dist="he" if dist == "normal" else dist,
                            bias=("normal:0.1" if dist == "normal" else dist) if bias else None, seed=seed,
                            groups=groups)
    x, wt, b = workloads.make_inputs(wl)
    return wl, x, wt, b


def _check(sg, wl, x, w, b, algo, what):
    got = gpu_conv(sg, x, w, b, wl.options(), algo=algo)
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    check_close(got, ref, wl.c // wl.groups, wl.r, wl.s, what)
    return got


@pytest.mark.parametrize("geom", [
    dict(n=2, h=14, w=14, c=128, k=128, r=3, s=3, groups=2, pad=1),            # C/G = 64: TMA im2col
    dict(n=2, h=12, w=12, c=512, k=256, r=3, s=3, groups=4, pad=1),            # C/G = 128, K/G = 64
    dict(n=2, h=10, w=10, c=128, k=192, r=3, s=3, groups=2, pad=1),            # K/G = 96: ragged column block
    dict(n=4, h=16, w=16, c=256, k=256, r=3, s=3, groups=32, stride=2, pad=1), # C/G = 8: cp.async (ResNeXt-like)
    dict(n=2, h=9, w=11, c=64, k=32, r=3, s=3, groups=4, pad=1, dil=2),        # C/G = 16, K/G = 8
    dict(n=2, h=12, w=12, c=16, k=16, r=3, s=3, groups=16, pad=1),             # depthwise: scalar gather
    dict(n=1, h=7, w=7, c=24, k=48, r=3, s=3, groups=3, pad=1),                # C/G = 8, K/G = 16
    dict(n=2, h=8, w=8, c=192, k=96, r=1, s=1, groups=3),                      # grouped 1x1, C/G = 64
])
def test_grouped_geometries(sg, geom):
    kw = dict(geom)
    wl, x, w, b = _case(kw.pop("n"), kw.pop("h"), kw.pop("w"), kw.pop("c"), kw.pop("k"), kw.pop("r"), kw.pop("s"),
                        kw.pop("groups"), seed=31, **kw)
    _check(sg, wl, x, w, b, make_algo(sg, wait_limit_ns=WAIT), wl.describe())


@pytest.mark.parametrize("loader", [1, 2, 3])
@pytest.mark.parametrize("bn", [64, 128])
def test_each_loader_and_width(sg, loader, bn):
    # C/G = 64, K/G = 96: every loader that can run grouped work, both tile widths.
    wl, x, w, b = _case(2, 10, 10, 128, 192, 3, 3, 2, pad=1, seed=32)
    _check(sg, wl, x, w, b, make_algo(sg, loader=loader, block_n=bn, wait_limit_ns=WAIT),
           f"groups loader={loader} bn={bn}")


@pytest.mark.parametrize("algo_kw", [dict(splits=3), dict(splits=3, reduction=1), dict(grid=5), dict(grid=13)])
def test_split_and_stream_k(sg, algo_kw):
    # Cut tiles of a grouped problem reduce in place per group.
    wl, x, w, b = _case(2, 8, 8, 256, 128, 3, 3, 2, pad=1, seed=33)
    _check(sg, wl, x, w, b, make_algo(sg, wait_limit_ns=WAIT, **algo_kw), f"groups {algo_kw}")


def test_integer_inputs_exact(sg):
    wl, x, w, b = _case(2, 9, 9, 128, 64, 3, 3, 2, pad=1, seed=34, dist="int:-3:3")
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, wait_limit_ns=WAIT))
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    assert np.array_equal(got.astype(np.float64), ref)


def test_groups_match_separate_convolutions(sg):
    # Grouped result = concatenation of ordinary convolutions on each group's channels.
    wl, x, w, b = _case(2, 10, 10, 128, 128, 3, 3, 2, pad=1, seed=35)
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, wait_limit_ns=WAIT))
    opts = dict(wl.options(), groups=1)
    parts = [gpu_conv(sg, x[..., g * 64:(g + 1) * 64].contiguous(), w[g * 64:(g + 1) * 64].contiguous(),
                      b[g * 64:(g + 1) * 64].contiguous(), opts, algo=make_algo(sg, wait_limit_ns=WAIT))
             for g in range(2)]
    check_close(got, np.concatenate(parts, axis=-1).astype(np.float64), 64, 3, 3, "groups vs separate")


def test_box_halo_and_row_window_refuse_groups(sg):
    import split_gemm_gb300 as m
    wl, x, w, b = _case(1, 8, 8, 256, 128, 3, 3, 2, pad=1, seed=36)
    for loader in (5, 6, 7):
        with pytest.raises(m.Conv2dError):
            gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=loader))


@pytest.mark.parametrize("name", sorted(workloads.GROUPED))
def test_grouped_workload_full_size(sg, name):
    wl = workloads.get(name)
    x, w, b = workloads.make_inputs(wl)
    _check(sg, wl, x, w, b, None, name)
