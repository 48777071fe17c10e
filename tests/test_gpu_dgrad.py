"""Data gradient (conv2d_bwd_data) and conv_transpose2d against the CPU oracle, element
by element, through the C ABI (needs a GB300): stride 1 (one launch) and strides 2 and 3
(one launch per output phase, the sub-pixel decomposition).

Inputs: dy ~ N(0, 1), weights He-init as the forward workloads draw them, so each
term dy*w has the forward terms' scale and the forward bar applies with C*R*S
replaced by the data gradient's reduction length K*R*S:
|gpu - ref| <= 1e-5*|ref| + 1e-4*sqrt(K*R*S).  Integer inputs must match exactly."""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import dgrad as od
from tests.parity import check_close, make_algo

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


def _extent(i, pad, dil, ker, st):
    room = i + 2 * pad - (dil * (ker - 1) + 1)
    return 0 if room < 0 else room // st + 1


def _case(n, h, w, c, k, r, s, pad=0, dil=1, seed=0, ints=False, stride=1):
    def pair(v):
        return v if isinstance(v, tuple) else (v, v)
    (ph, pw), (dh, dw), (sh, sw) = pair(pad), pair(dil), pair(stride)
    p, q = _extent(h, ph, dh, r, sh), _extent(w, pw, dw, s, sw)
    g = torch.Generator().manual_seed(2000 + seed)
    if ints:
        dy = torch.randint(-3, 4, (n, p, q, k), generator=g).to(torch.bfloat16)
        wt = torch.randint(-3, 4, (k, r, s, c), generator=g).to(torch.bfloat16)
    else:
        dy = torch.randn((n, p, q, k), generator=g).to(torch.bfloat16)
        wt = (torch.randn((k, r, s, c), generator=g) * math.sqrt(2.0 / (c * r * s))).to(torch.bfloat16)
    opts = dict(stride=(sh, sw), padding=(ph, pw), dilation=(dh, dw))
    return dy, wt, (n, h, w, c), opts


def _gpu(sg, dy, wt, x_shape, opts, algo=None, workspace=None):
    dev = torch.device("cuda", 0)
    dx = torch.full(x_shape, float("nan"), dtype=torch.float32, device=dev)
    sg.conv2d_bwd_data_into(dx, dy.to(dev), wt.to(dev), **opts, algo=algo, workspace=workspace)
    torch.cuda.synchronize()
    return dx.cpu().numpy()


GEOMS = [
    ("3x3_pad1", dict(n=2, h=14, w=14, c=64, k=64, r=3, s=3, pad=1)),
    ("c96_ragged_cols", dict(n=2, h=10, w=12, c=96, k=128, r=3, s=3, pad=1)),
    ("dil2_pad2", dict(n=2, h=12, w=11, c=128, k=64, r=3, s=3, pad=2, dil=2)),
    ("asym_3x2", dict(n=3, h=9, w=10, c=64, k=64, r=3, s=2, pad=(0, 1))),
    ("valid_pad0", dict(n=2, h=9, w=9, c=64, k=128, r=3, s=3, pad=0)),
    ("1x1", dict(n=2, h=16, w=16, c=256, k=128, r=1, s=1)),
    ("7x7_pad3", dict(n=1, h=20, w=20, c=64, k=64, r=7, s=7, pad=3)),
    ("c8_tiny", dict(n=2, h=6, w=7, c=8, k=64, r=3, s=3, pad=1)),
    ("ragged_m", dict(n=3, h=13, w=11, c=72, k=192, r=3, s=3, pad=1)),
]


@pytest.mark.parametrize("bn", [0, 64, 128, 256])
@pytest.mark.parametrize("geom", GEOMS, ids=[g[0] for g in GEOMS])
def test_dgrad_geometries(sg, geom, bn):
    name, kw = geom
    kw = dict(kw)
    k, r, s = kw["k"], kw["r"], kw["s"]
    dy, wt, xs, opts = _case(kw.pop("n"), kw.pop("h"), kw.pop("w"), kw.pop("c"), kw.pop("k"), kw.pop("r"),
                             kw.pop("s"), seed=zlib.crc32(name.encode()) % 1000, **kw)
    got = _gpu(sg, dy, wt, xs, opts, algo=make_algo(sg, block_n=bn, wait_limit_ns=WAIT))
    assert sg.last_launch_count() == 1
    ref = od.conv2d_dgrad(dy, wt, xs, **opts)
    check_close(got, ref, k, r, s, f"dgrad {name} bn={bn}")


@pytest.mark.parametrize("forced", [dict(splits=1), dict(splits=3), dict(splits=9), dict(grid=7), dict(grid=50),
                                    dict(splits=4, reduction=1), dict(grid=23, reduction=1)],
                         ids=["splits1", "splits3", "splits9", "grid7", "grid50", "splits4_ordered",
                              "grid23_ordered"])
def test_dgrad_forced_plans(sg, forced):
    dy, wt, xs, opts = _case(2, 9, 9, 128, 256, 3, 3, pad=1, seed=4)  # 36 k-blocks of 64
    params = sg.make_params(xs, wt.shape, **opts)
    ws = torch.zeros(sg.dgrad_workspace_bytes(params), dtype=torch.uint8, device="cuda")
    got = _gpu(sg, dy, wt, xs, opts, algo=make_algo(sg, wait_limit_ns=WAIT, **forced), workspace=ws)
    ref = od.conv2d_dgrad(dy, wt, xs, **opts)
    check_close(got, ref, 256, 3, 3, f"dgrad forced {forced}")
    assert int(torch.count_nonzero(ws)) == 0
    assert sg.status(ws) == 0


@pytest.mark.parametrize("bn", [64, 128, 256])
def test_dgrad_integer_inputs_exact(sg, bn):
    dy, wt, xs, opts = _case(2, 11, 13, 128, 128, 3, 3, pad=(1, 2), dil=(1, 2), seed=7, ints=True)
    got = _gpu(sg, dy, wt, xs, opts, algo=make_algo(sg, block_n=bn, wait_limit_ns=WAIT))
    ref = od.conv2d_dgrad(dy, wt, xs, **opts)
    assert np.array_equal(got, ref), f"{int(np.count_nonzero(got != ref))} of {got.size} differ"


@pytest.mark.parametrize("geom", [(2, 9, 9, 64, 64, 3, 3, 1, 1), (1, 12, 10, 128, 96, 3, 3, 0, 1),
                                  (2, 8, 8, 64, 64, 3, 3, 2, 2), (1, 7, 9, 64, 32, 5, 3, 2, 1)])
def test_conv_transpose2d_stride1(sg, geom):
    """conv_transpose2d(x, w) of x [N,Hi,Wi,Cin], w [Cin,R,S,Cout] equals the data gradient
    with dy = x (the oracle's definition, pinned against torch's gradient)."""
    n, hi, wi, cin, cout, r, s, pad, dil = geom
    g = torch.Generator().manual_seed(sum(geom))
    x = torch.randn((n, hi, wi, cin), generator=g).to(torch.bfloat16)
    wt = (torch.randn((cin, r, s, cout), generator=g) * math.sqrt(2.0 / (cin * r * s))).to(torch.bfloat16)
    y = sg.conv_transpose2d(x.cuda(), wt.cuda(), padding=pad, dilation=dil)
    torch.cuda.synchronize()
    ho, wo = hi - 2 * pad + dil * (r - 1), wi - 2 * pad + dil * (s - 1)
    assert tuple(y.shape) == (n, ho, wo, cout)
    ref = od.conv2d_dgrad(x, wt, (n, ho, wo, cout), 1, pad, dil)
    check_close(y.cpu().numpy(), ref, cin, r, s, f"conv_transpose2d {geom}")


def test_dgrad_no_filters_gives_zero(sg):
    dev = torch.device("cuda", 0)
    dy = torch.zeros((2, 6, 6, 0), dtype=torch.bfloat16, device=dev)
    wt = torch.zeros((0, 3, 3, 64), dtype=torch.bfloat16, device=dev)
    dx = sg.conv2d_bwd_data(dy, wt, (2, 6, 6, 64), padding=1)
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(dx)) == 0


@pytest.mark.parametrize("xs,ws,stride,pad,groups", [
    ((1, 8, 8, 64), (64, 3, 3, 64), 2, 2, 1),   # stride 2, pad 2: phase 1 has one tap and padding -1
    ((1, 8, 8, 64), (32, 3, 3, 64), 1, 1, 1),   # K % 64 != 0
    ((1, 8, 8, 12), (64, 3, 3, 12), 1, 1, 1),   # C % 8 != 0
    ((1, 8, 8, 128), (64, 3, 3, 64), 1, 1, 2),  # groups
    ((1, 8, 8, 64), (64, 3, 3, 64), 1, 3, 1),   # pad > dil*(R-1)
])
def test_dgrad_unsupported_shapes_refused(sg, xs, ws, stride, pad, groups):
    dev = torch.device("cuda", 0)
    p = _extent(xs[1], pad, 1, ws[1], stride)
    dy = torch.zeros((xs[0], p, p, ws[0]), dtype=torch.bfloat16, device=dev)
    wt = torch.zeros(ws, dtype=torch.bfloat16, device=dev)
    with pytest.raises(sg.Conv2dError) as e:
        sg.conv2d_bwd_data(dy, wt, xs, stride=stride, padding=pad, groups=groups)
    assert e.value.code == 2


def _phases_with_taps(h, st, pad, dil, ker):
    """Output phases a (rows h = a + st*i exist) that some filter tap reaches."""
    return [a for a in range(min(st, h)) if any((a + pad - r * dil) % st == 0 for r in range(ker))]


STRIDED = [
    ("s2_3x3_pad1", dict(n=2, h=14, w=14, c=64, k=64, r=3, s=3, pad=1, stride=2)),
    ("s2_1x1", dict(n=2, h=15, w=16, c=128, k=64, r=1, s=1, pad=0, stride=2)),      # phases with no tap
    ("s2_7x7_pad3", dict(n=1, h=22, w=20, c=64, k=64, r=7, s=7, pad=3, stride=2)),
    ("s2_dil2", dict(n=2, h=13, w=12, c=64, k=128, r=3, s=3, pad=2, dil=2, stride=2)),  # gcd(2, 2) = 2
    ("s3_5x3", dict(n=2, h=17, w=16, c=72, k=64, r=5, s=3, pad=(2, 0), stride=3)),
    ("s23_asym", dict(n=3, h=11, w=13, c=64, k=192, r=3, s=4, pad=(1, 1), stride=(2, 3))),
    ("s2_valid", dict(n=2, h=9, w=10, c=96, k=64, r=3, s=3, pad=0, stride=2)),
    ("s2_ragged_h", dict(n=1, h=7, w=9, c=8, k=64, r=4, s=2, pad=(1, 0), stride=(3, 2))),
]


@pytest.mark.parametrize("bn", [0, 64, 256])
@pytest.mark.parametrize("geom", STRIDED, ids=[g[0] for g in STRIDED])
def test_dgrad_strided_geometries(sg, geom, bn):
    """Stride > 1: one launch per output phase that a tap reaches; the rest of dx is zero."""
    name, kw = geom
    kw = dict(kw)
    def pair(v):
        return v if isinstance(v, tuple) else (v, v)
    k, r, s = kw["k"], kw["r"], kw["s"]
    (sh, sw), (ph, pw), (dh, dw) = pair(kw["stride"]), pair(kw["pad"]), pair(kw.get("dil", 1))
    dy, wt, xs, opts = _case(kw.pop("n"), kw.pop("h"), kw.pop("w"), kw.pop("c"), kw.pop("k"), kw.pop("r"),
                             kw.pop("s"), seed=zlib.crc32(name.encode()) % 1000, **kw)
    got = _gpu(sg, dy, wt, xs, opts, algo=make_algo(sg, block_n=bn, wait_limit_ns=WAIT))
    phases = len(_phases_with_taps(xs[1], sh, ph, dh, r)) * len(_phases_with_taps(xs[2], sw, pw, dw, s))
    assert sg.last_launch_count() == phases
    ref = od.conv2d_dgrad(dy, wt, xs, **opts)
    check_close(got, ref, k, r, s, f"dgrad {name} bn={bn}")


@pytest.mark.parametrize("stride,pad", [(2, 1), (3, 0)])
def test_dgrad_strided_integer_inputs_exact(sg, stride, pad):
    dy, wt, xs, opts = _case(2, 13, 14, 64, 128, 3, 3, pad=pad, seed=17 + stride, ints=True, stride=stride)
    got = _gpu(sg, dy, wt, xs, opts, algo=make_algo(sg, wait_limit_ns=WAIT))
    ref = od.conv2d_dgrad(dy, wt, xs, **opts)
    assert np.array_equal(got, ref), f"{int(np.count_nonzero(got != ref))} of {got.size} differ"


@pytest.mark.parametrize("forced", [dict(splits=3), dict(grid=3), dict(splits=2, reduction=1)],
                         ids=["splits3", "grid3", "splits2_ordered"])
def test_dgrad_strided_cut_tiles(sg, forced):
    """Cut tiles in every phase (the one-tap phase has 4 k-blocks), the phases reusing one
    workspace in stream order."""
    dy, wt, xs, opts = _case(2, 12, 12, 128, 256, 3, 3, pad=1, seed=9, stride=2)
    params = sg.make_params(xs, wt.shape, **opts)
    ws = torch.zeros(sg.dgrad_workspace_bytes(params), dtype=torch.uint8, device="cuda")
    got = _gpu(sg, dy, wt, xs, opts, algo=make_algo(sg, wait_limit_ns=WAIT, **forced), workspace=ws)
    ref = od.conv2d_dgrad(dy, wt, xs, **opts)
    check_close(got, ref, 256, 3, 3, f"strided dgrad forced {forced}")
    assert int(torch.count_nonzero(ws)) == 0
    assert sg.status(ws) == 0


@pytest.mark.parametrize("geom", [(2, 7, 7, 64, 64, 3, 3, 1, 1, 2, 1), (1, 6, 5, 64, 32, 4, 4, 1, 1, 2, 0),
                                  (2, 5, 6, 128, 64, 3, 3, 0, 1, 3, 2)])
def test_conv_transpose2d_strided(sg, geom):
    """conv_transpose2d with stride and output padding: the data gradient of the forward
    conv from the transposed output size back to the input's (oracle definition)."""
    n, hi, wi, cin, cout, r, s, pad, dil, st, op = geom
    g = torch.Generator().manual_seed(sum(geom))
    x = torch.randn((n, hi, wi, cin), generator=g).to(torch.bfloat16)
    wt = (torch.randn((cin, r, s, cout), generator=g) * math.sqrt(2.0 / (cin * r * s))).to(torch.bfloat16)
    y = sg.conv_transpose2d(x.cuda(), wt.cuda(), padding=pad, dilation=dil, stride=st, output_padding=op)
    torch.cuda.synchronize()
    ho = (hi - 1) * st - 2 * pad + dil * (r - 1) + 1 + op
    wo = (wi - 1) * st - 2 * pad + dil * (s - 1) + 1 + op
    assert tuple(y.shape) == (n, ho, wo, cout)
    ref = od.conv2d_dgrad(x, wt, (n, ho, wo, cout), st, pad, dil)
    check_close(y.cpu().numpy(), ref, cin, r, s, f"conv_transpose2d {geom}")


FULL = ["resnet_56x56_c64", "resnet_28x28_c256", "splitk_7x7_c2048", "dil2_64_c128", "proj_56_c256_1x1s2"]


@pytest.mark.parametrize("name", FULL)
def test_dgrad_full_size_workloads(sg, name):
    """The data gradient of each eligible workload at full size (the heuristic's plan; the
    1x1 stride-2 projection through its one phase with a tap, the other three zero), checked
    on sampled elements against the oracle one by one."""
    wl = workloads.get(name)
    _, w, _ = workloads.make_inputs(wl)
    dy = workloads.make_output_grad(wl, variance=1.0)
    o = wl.options()
    xs = (wl.n, wl.h, wl.w, wl.c)
    got = _gpu(sg, dy, w, xs, dict(stride=o["stride"], padding=o["padding"], dilation=o["dilation"]))
    assert sg.last_launch_count() == 1  # stride 1, or one phase with a tap
    flat = got.reshape(-1, wl.c)
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    mi = np.concatenate([rng.integers(0, flat.shape[0], 3000), [0, 0, flat.shape[0] - 1, flat.shape[0] - 1]])
    ci = np.concatenate([rng.integers(0, wl.c, 3000), [0, wl.c - 1, 0, wl.c - 1]])
    ref, _ = od.conv2d_dgrad_points_f64(oracle.widen_bf16(dy), oracle.widen_bf16(w), xs, o["stride"], o["padding"],
                                        o["dilation"], mi, ci)
    check_close(flat[mi, ci], ref, wl.k, wl.r, wl.s, f"dgrad {name}")
    assert np.all(np.isfinite(flat)), f"{name}: an input-gradient element was not written"
