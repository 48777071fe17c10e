"""CUDA path vs the CPU oracle, element by element, through the C ABI (needs a GB300)."""
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


def _case(n, h, w, c, k, r, s, stride=1, pad=0, dil=1, bias=True, seed=0, dist="normal"):
    def pair(v):
        return v if isinstance(v, tuple) else (v, v)
    (sh, sw), (ph, pw), (dh, dw) = pair(stride), pair(pad), pair(dil)
    wl = workloads.Workload(f"case{seed}", n, h, w, c, k, r, s, sh, sw, ph, pw, dh, dw,
                            x_dist=dist, w_dist="he" if dist == "normal" else dist,
                            bias=("normal:0.1" if dist == "normal" else dist) if bias else None, seed=seed)
    x, wt, b = workloads.make_inputs(wl)
    return wl, x, wt, b


def _run_and_check(sg, wl, x, w, b, algo=None, what=""):
    got = gpu_conv(sg, x, w, b, wl.options(), algo=algo)
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    check_close(got, ref, wl.c, wl.r, wl.s, what or wl.describe())
    return got


# ---------------------------------------------------------------- loaders on small shapes
def test_tiny_workload_default(sg):
    wl = workloads.get("tiny_8x8_c16")
    x, w, b = workloads.make_inputs(wl)
    _run_and_check(sg, wl, x, w, b)


@pytest.mark.parametrize("loader", [2, 3])
def test_tiny_workload_gather_loaders(sg, loader):
    wl = workloads.get("tiny_8x8_c16")
    x, w, b = workloads.make_inputs(wl)
    _run_and_check(sg, wl, x, w, b, make_algo(sg, loader=loader, wait_limit_ns=WAIT))


@pytest.mark.parametrize("loader", [1, 2, 3, 4])
@pytest.mark.parametrize("bn", [64, 128, 256])
def test_c64_each_loader_each_width(sg, loader, bn):
    # 2 images of 10x10, 3x3 pad 1: M = 200 (one full tile + a ragged tail), K = 80 (ragged in N).
    wl, x, w, b = _case(2, 10, 10, 64, 80, 3, 3, pad=1, seed=1)
    _run_and_check(sg, wl, x, w, b, make_algo(sg, block_n=bn, loader=loader, wait_limit_ns=WAIT),
                   f"loader={loader} bn={bn}")


@pytest.mark.parametrize("bn", [64, 128, 256])
@pytest.mark.parametrize("grid", [0, 1, 3])
def test_256_pixel_tiles(sg, bn, grid):
    # M = 3*10*10 = 300: one full 256-row tile and a ragged one; K = 200 ragged in N.
    # grid 1 and 3 put several tiles (and cut tiles) on one CTA.
    wl, x, w, b = _case(3, 10, 10, 64, 200, 3, 3, pad=1, seed=4)
    _run_and_check(sg, wl, x, w, b, make_algo(sg, block_m=256, block_n=bn, loader=1, grid=grid, wait_limit_ns=WAIT),
                   f"BM=256 bn={bn} grid={grid}")


@pytest.mark.parametrize("geom", [
    dict(stride=(2, 1), pad=(1, 0), dil=1),
    dict(stride=1, pad=(2, 1), dil=(2, 1)),
    dict(stride=(1, 3), pad=(0, 2), dil=(1, 2)),
    dict(stride=2, pad=3, dil=1),
])
@pytest.mark.parametrize("loader", [1, 2, 4])
def test_asymmetric_windows(sg, geom, loader):
    wl, x, w, b = _case(2, 13, 11, 64, 64, 3, 5, seed=2, **geom)
    _run_and_check(sg, wl, x, w, b, make_algo(sg, loader=loader, wait_limit_ns=WAIT), f"{geom} loader={loader}")


@pytest.mark.parametrize("seed", range(16))
def test_random_small_default_heuristic(sg, seed):
    wl = workloads.random_small(seed, max_hw=14)
    x, w, b = workloads.make_inputs(wl)
    _run_and_check(sg, wl, x, w, b)


@pytest.mark.parametrize("seed", range(6))
def test_random_small_integer_inputs_scalar_loader(sg, seed):
    # Small integer inputs: every partial sum is exact in fp32, so the result is exact.
    wl = workloads.random_small(100 + seed, max_hw=12, ints=True)
    x, w, b = workloads.make_inputs(wl)
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=3, wait_limit_ns=WAIT))
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    assert np.array_equal(got.astype(np.float64), ref), wl.describe()


# ---------------------------------------------------------------- edge cases
@pytest.mark.parametrize("shape", [
    dict(n=1, h=1, w=1, c=8, k=16, r=1, s=1),             # M = 1
    dict(n=3, h=5, w=7, c=1, k=5, r=3, s=3, pad=1),       # C = 1, K % 4 != 0 (no TMA store)
    dict(n=1, h=9, w=9, c=3, k=130, r=3, s=3, pad=1),     # C = 3, K beyond one 128 tile
    dict(n=2, h=7, w=1, c=24, k=32, r=7, s=1, pad=3),     # W = 1, tall filter
    dict(n=1, h=4, w=4, c=512, k=64, r=3, s=3, pad=1),    # long reduction on few pixels
    dict(n=5, h=3, w=3, c=64, k=8, r=3, s=3),             # P = Q = 1
])
def test_edge_shapes(sg, shape):
    kw = dict(shape)
    wl, x, w, b = _case(kw.pop("n"), kw.pop("h"), kw.pop("w"), kw.pop("c"), kw.pop("k"), kw.pop("r"), kw.pop("s"),
                        seed=3, **kw)
    _run_and_check(sg, wl, x, w, b)


def test_empty_batch_is_a_no_op(sg):
    x = torch.zeros((0, 8, 8, 16), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((16, 3, 3, 16), dtype=torch.bfloat16, device="cuda")
    y = sg.conv2d_fwd(x, w, None, padding=1)
    torch.cuda.synchronize()
    assert tuple(y.shape) == (0, 8, 8, 16)
    assert sg.last_launch_count() == 0


def test_forced_tma_loader_rejects_small_channels(sg):
    wl = workloads.get("tiny_8x8_c16")
    x, w, b = workloads.make_inputs(wl)
    with pytest.raises(sg.Conv2dError) as e:
        gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=1))
    assert e.value.code == 2


def test_misaligned_pointer_rejected_before_launch(sg):
    base = torch.zeros(1 * 8 * 8 * 16 + 1, dtype=torch.bfloat16, device="cuda")
    x = base[1:].view(1, 8, 8, 16)  # 2-byte offset
    w = torch.zeros((16, 3, 3, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sg.Conv2dError) as e:
        sg.conv2d_fwd(x, w, None, padding=1)
    assert e.value.code == 3


def test_groups_that_do_not_divide_rejected(sg):
    # groups must divide both C and K (CONV2D_ERR_INVALID); a dividing value runs.
    x = torch.zeros((1, 8, 8, 18), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((16, 3, 3, 6), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sg.Conv2dError) as e:
        sg.conv2d_fwd(x, w, None, padding=1, groups=3)  # C = 18 divides, K = 16 does not
    assert e.value.code == 1
    y = sg.conv2d_fwd(x[..., :16].contiguous(), torch.zeros((16, 3, 3, 8), dtype=torch.bfloat16, device="cuda"),
                      None, padding=1, groups=2)
    torch.cuda.synchronize()
    assert y.shape == (1, 8, 8, 16) and not bool(y.abs().sum())
