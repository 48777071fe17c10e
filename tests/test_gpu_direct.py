"""The direct (CUDA-core) kernel for groups of few channels -- C/groups = K/groups in
{1, 2, 4, 8, 16}, depthwise included -- against the CPU oracle, element by element,
through the C ABI (needs a GB300).  Where block-diagonal tensor-core tiles apply
(C/groups in {8, 16, 32}) the heuristic takes those instead; these tests force the
direct kernel."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import epilogue
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
    wl = workloads.Workload(f"dir{seed}", n, h, w, c, k, r, s, sh, sw, ph, pw, dh, dw,
                            x_dist=dist, w_dist="he" if dist == "normal" else dist,
                            bias=("normal:0.1" if dist == "normal" else dist) if bias else None, seed=seed,
                            groups=groups)
    x, wt, b = workloads.make_inputs(wl)
    return wl, x, wt, b


GEOMS = [
    ("resnext_cg8", dict(n=2, h=14, w=14, c=256, k=256, r=3, s=3, groups=32, pad=1)),
    ("depthwise_s2", dict(n=2, h=15, w=13, c=64, k=64, r=3, s=3, groups=64, stride=2, pad=1)),
    ("depthwise_7x7", dict(n=1, h=20, w=20, c=96, k=96, r=7, s=7, groups=96, pad=3, bias=False)),
    ("cg2_dil2", dict(n=2, h=12, w=11, c=32, k=32, r=3, s=3, groups=16, pad=2, dil=2)),
    ("cg4_asym", dict(n=3, h=9, w=10, c=64, k=64, r=3, s=2, groups=16, stride=(2, 1), pad=(1, 0))),
    ("cg16", dict(n=2, h=10, w=10, c=128, k=128, r=3, s=3, groups=8, pad=1)),
    ("cg8_1x1", dict(n=2, h=8, w=8, c=64, k=64, r=1, s=1, groups=8)),
    ("two_groups_cg8", dict(n=1, h=7, w=9, c=16, k=16, r=3, s=3, groups=2, pad=1)),
]


@pytest.mark.parametrize("geom", GEOMS, ids=[g[0] for g in GEOMS])
def test_direct_geometries(sg, geom):
    name, kw = geom
    kw = dict(kw)
    wl, x, w, b = _case(kw.pop("n"), kw.pop("h"), kw.pop("w"), kw.pop("c"), kw.pop("k"), kw.pop("r"), kw.pop("s"),
                        kw.pop("groups"), seed=51, **kw)
    params = sg.make_params(x.shape, w.shape, **wl.options())
    cg = wl.c // wl.groups
    bd = cg in (8, 16, 32) and wl.groups % (64 // cg) == 0  # block-diagonal tiles take these layers
    assert sg.query_algo(params).loader == (sg.LOADER_BLOCKDIAG if bd else sg.LOADER_DIRECT)
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=sg.LOADER_DIRECT))
    assert sg.last_launch_count() == 1
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    check_close(got, ref, wl.c // wl.groups, wl.r, wl.s, f"direct {name}")


@pytest.mark.parametrize("groups,c", [(32, 256), (64, 64), (16, 64), (8, 128)])
def test_direct_integer_inputs_exact(sg, groups, c):
    wl, x, w, b = _case(2, 9, 11, c, c, 3, 3, groups, pad=1, seed=52, dist="int:-3:3")
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=sg.LOADER_DIRECT))
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    assert np.array_equal(got, ref), f"{int(np.count_nonzero(got != ref))} of {got.size} differ"


@pytest.mark.parametrize("mode", [(True, False), (False, True), (True, True)], ids=["relu", "bf16", "relu_bf16"])
def test_direct_fused_epilogue(sg, mode):
    wl, x, w, b = _case(2, 14, 14, 256, 256, 3, 3, 32, pad=1, seed=53)
    direct = make_algo(sg, loader=sg.LOADER_DIRECT)
    got = gpu_conv_epi(sg, x, w, b, wl.options(), *mode, algo=direct)
    u = oracle.conv2d_fwd(x, w, b, **wl.options())
    check_epilogue(got, u, wl.c // wl.groups, wl.r, wl.s, *mode, "direct fused")
    # Same kernel, same summation order: the fused output is the plain one put through the epilogue.
    plain = gpu_conv_epi(sg, x, w, b, wl.options(), False, False, algo=direct)
    assert np.array_equal(got, epilogue.apply(plain, *mode))


def test_forced_gemm_loaders_still_run_small_groups(sg):
    """Forcing an implicit-GEMM loader keeps the tensor-core path for these shapes."""
    wl, x, w, b = _case(2, 10, 10, 256, 256, 3, 3, 32, pad=1, seed=54)
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    for loader in (2, 3):
        got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=loader))
        check_close(got, ref, 8, 3, 3, f"loader {loader}")
    # Forcing only a split also keeps the GEMM path (the direct kernel has no splits).
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, splits=2))
    check_close(got, ref, 8, 3, 3, "split 2")


@pytest.mark.parametrize("shape,groups", [(((1, 8, 8, 64), (64, 3, 3, 16)), 4),    # C/G = K/G = 16: eligible
                                          (((1, 8, 8, 48), (48, 3, 3, 3)), 16),    # C/G = 3
                                          (((1, 8, 8, 64), (64, 3, 3, 64)), 1)])   # groups == 1
def test_direct_refuses_ineligible_shapes(sg, shape, groups):
    xs, ws = shape
    x = torch.zeros(xs, dtype=torch.bfloat16)
    w = torch.zeros(ws, dtype=torch.bfloat16)
    params = sg.make_params(xs, ws, 1, 1, 1, groups)
    cg = xs[3] // groups
    eligible = (ws[0] // groups == cg and cg in (1, 2, 4, 8, 16) and groups > 1
                and xs[3] % (16 if cg == 16 else 8) == 0)
    if eligible:
        got = gpu_conv(sg, x, w, None, dict(stride=1, padding=1, dilation=1, groups=groups),
                       algo=make_algo(sg, loader=sg.LOADER_DIRECT))
        assert np.array_equal(got, np.zeros_like(got))
        return
    with pytest.raises(sg.Conv2dError) as e:
        gpu_conv(sg, x, w, None, dict(stride=1, padding=1, dilation=1, groups=groups),
                 algo=make_algo(sg, loader=sg.LOADER_DIRECT))
    assert e.value.code == 2
    assert sg.query_algo(params).loader != sg.LOADER_DIRECT
