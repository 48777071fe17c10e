"""Block-diagonal tensor-core tiles for grouped convolution (C/groups = K/groups = cg in
{8, 16, 32}): 64/cg groups merged into one 64-channel group whose weight, expanded into
the workspace with zeros outside each output channel's own group, feeds the grouped
implicit GEMM.  Against the CPU oracle (the grouped definition), element by element,
through the C ABI (needs a GB300)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import check_close, check_epilogue, gpu_conv, gpu_conv_epi, make_algo

pytestmark = pytest.mark.gpu


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
    wl = workloads.Workload(f"bd{seed}", n, h, w, c, k, r, s, sh, sw, ph, pw, dh, dw,
                            x_dist=dist, w_dist="he" if dist == "normal" else dist,
                            bias=("normal:0.1" if dist == "normal" else dist) if bias else None, seed=seed,
                            groups=groups)
    x, wt, b = workloads.make_inputs(wl)
    return wl, x, wt, b


GEOMS = [
    ("cg8_g32", dict(n=2, h=14, w=14, c=256, k=256, r=3, s=3, groups=32, pad=1)),
    ("cg8_g8_one_block", dict(n=2, h=9, w=11, c=64, k=64, r=3, s=3, groups=8, pad=1)),
    ("cg16_g8", dict(n=2, h=10, w=10, c=128, k=128, r=3, s=3, groups=8, pad=1)),
    ("cg32_g4", dict(n=2, h=12, w=9, c=128, k=128, r=3, s=3, groups=4, pad=1)),
    ("cg8_stride2", dict(n=3, h=15, w=13, c=128, k=128, r=3, s=3, groups=16, stride=2, pad=1)),
    ("cg16_dil2_asym", dict(n=2, h=12, w=11, c=64, k=64, r=3, s=2, groups=4, pad=(2, 1), dil=2)),
    ("cg8_1x1", dict(n=2, h=8, w=8, c=64, k=64, r=1, s=1, groups=8, bias=False)),
    ("cg32_5x5", dict(n=1, h=11, w=12, c=64, k=64, r=5, s=5, groups=2, pad=2)),
]


@pytest.mark.parametrize("geom", GEOMS, ids=[g[0] for g in GEOMS])
def test_blockdiag_geometries(sg, geom):
    name, kw = geom
    kw = dict(kw)
    wl, x, w, b = _case(kw.pop("n"), kw.pop("h"), kw.pop("w"), kw.pop("c"), kw.pop("k"), kw.pop("r"), kw.pop("s"),
                        kw.pop("groups"), seed=61, **kw)
    params = sg.make_params(x.shape, w.shape, **wl.options())
    assert sg.query_algo(params).loader == sg.LOADER_BLOCKDIAG
    got = gpu_conv(sg, x, w, b, wl.options())
    assert sg.last_launch_count() == 2  # the weight expansion and the convolution
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    check_close(got, ref, wl.c // wl.groups, wl.r, wl.s, f"block-diagonal {name}")


def test_blockdiag_leaves_the_workspace_zero(sg):
    """The expanded weight lives in the workspace only during the call: the workspace is
    zero afterwards (a later call's semaphores and partial sums assume it)."""
    wl, x, w, b = _case(2, 10, 10, 256, 256, 3, 3, 32, pad=1, seed=65)
    params = sg.make_params(x.shape, w.shape, **wl.options())
    ws = torch.zeros(sg.workspace_bytes(params), dtype=torch.uint8, device="cuda")
    got = gpu_conv(sg, x, w, b, wl.options(), workspace=ws)
    assert sg.last_launch_count() == 2
    check_close(got, oracle.conv2d_fwd(x, w, b, **wl.options()), 8, 3, 3, "block-diagonal")
    assert int(torch.count_nonzero(ws)) == 0


@pytest.mark.parametrize("groups,c", [(32, 256), (8, 128), (4, 128)])
def test_blockdiag_integer_inputs_exact(sg, groups, c):
    """Small integers: the zero blocks add exact zeros, so the result equals the oracle's."""
    wl, x, w, b = _case(2, 9, 11, c, c, 3, 3, groups, pad=1, seed=62, dist="int:-3:3")
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=sg.LOADER_BLOCKDIAG))
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    assert np.array_equal(got, ref), f"{int(np.count_nonzero(got != ref))} of {got.size} differ"


@pytest.mark.parametrize("mode", [(True, False), (False, True), (True, True)], ids=["relu", "bf16", "relu_bf16"])
def test_blockdiag_fused_epilogue(sg, mode):
    wl, x, w, b = _case(2, 14, 14, 256, 256, 3, 3, 32, pad=1, seed=63)
    got = gpu_conv_epi(sg, x, w, b, wl.options(), *mode)
    u = oracle.conv2d_fwd(x, w, b, **wl.options())
    check_epilogue(got, u, wl.c // wl.groups, wl.r, wl.s, *mode, "block-diagonal fused")


def test_blockdiag_small_workspace_takes_the_direct_kernel(sg):
    """A workspace without room for the expanded weight: the direct kernel runs instead (one
    launch), at parity; forcing the block-diagonal tiles then reports the missing room."""
    wl, x, w, b = _case(2, 10, 10, 128, 128, 3, 3, 16, pad=1, seed=64)
    params = sg.make_params(x.shape, w.shape, **wl.options())
    small = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    assert sg.workspace_bytes(params) > small.numel()
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    got = gpu_conv(sg, x, w, b, wl.options(), workspace=small)
    assert sg.last_launch_count() == 1
    check_close(got, ref, 8, 3, 3, "small workspace")
    with pytest.raises(sg.Conv2dError) as e:
        gpu_conv(sg, x, w, b, wl.options(), workspace=small, algo=make_algo(sg, loader=sg.LOADER_BLOCKDIAG))
    assert e.value.code == 4  # CONV2D_ERR_WORKSPACE


@pytest.mark.parametrize("shape,groups", [(((1, 8, 8, 48), (48, 3, 3, 8)), 6),     # 6 groups of 8: 6 % 8 != 0
                                          (((1, 8, 8, 64), (64, 3, 3, 4)), 16),    # cg = 4
                                          (((1, 8, 8, 64), (32, 3, 3, 16)), 4)])   # K/G != C/G
def test_blockdiag_refuses_ineligible_shapes(sg, shape, groups):
    xs, ws = shape
    x = torch.zeros(xs, dtype=torch.bfloat16)
    w = torch.zeros(ws, dtype=torch.bfloat16)
    with pytest.raises(sg.Conv2dError) as e:
        gpu_conv(sg, x, w, None, dict(stride=1, padding=1, dilation=1, groups=groups),
                 algo=make_algo(sg, loader=sg.LOADER_BLOCKDIAG))
    assert e.value.code == 2


@pytest.mark.parametrize("name", ["resnext_28x28_c256_g32"])
def test_blockdiag_full_size_workload(sg, name):
    wl = workloads.get(name)
    x, w, b = workloads.make_inputs(wl)
    got = gpu_conv(sg, x, w, b, wl.options())
    assert sg.last_launch_count() == 2
    flat = got.reshape(-1, wl.k)
    rng = np.random.default_rng(7)
    mi = np.concatenate([rng.integers(0, flat.shape[0], 3000), [0, flat.shape[0] - 1]])
    ki = np.concatenate([rng.integers(0, wl.k, 3000), [0, wl.k - 1]])
    o = wl.options()
    ref = oracle.conv2d_fwd_points(x, w, b, o["stride"], o["padding"], o["dilation"], mi, ki, groups=o["groups"])
    check_close(flat[mi, ki], ref, wl.c // wl.groups, wl.r, wl.s, name)
