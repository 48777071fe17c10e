"""Weight gradient (conv2d_bwd_weight) against the CPU oracle, element by element,
through the C ABI (needs a GB300).

Inputs: x as the forward workloads draw it, dy ~ N(0, 2/L) with L = N*P*Q the
reduction length of every gradient element (the He scaling the forward weights
use for their reduction), so the forward parity bar applies with C*R*S replaced
by L: |gpu - ref| <= 1e-5*|ref| + 1e-4*sqrt(L).  Integer inputs give exact fp32
sums and must match bit for bit."""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import wgrad as ow
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


def _case(n, h, w, c, k, r, s, stride=1, pad=0, dil=1, seed=0, ints=False):
    def pair(v):
        return v if isinstance(v, tuple) else (v, v)
    (sh, sw), (ph, pw), (dh, dw) = pair(stride), pair(pad), pair(dil)
    p, q = _extent(h, ph, dh, r, sh), _extent(w, pw, dw, s, sw)
    g = torch.Generator().manual_seed(1000 + seed)
    if ints:
        x = torch.randint(-3, 4, (n, h, w, c), generator=g).to(torch.bfloat16)
        dy = torch.randint(-3, 4, (n, p, q, k), generator=g).to(torch.bfloat16)
    else:
        x = torch.randn((n, h, w, c), generator=g).to(torch.bfloat16)
        dy = (torch.randn((n, p, q, k), generator=g) * math.sqrt(2.0 / max(1, n * p * q))).to(torch.bfloat16)
    opts = dict(stride=(sh, sw), padding=(ph, pw), dilation=(dh, dw))
    return x, dy, (k, r, s, c), opts, n * p * q


def _gpu(sg, x, dy, w_shape, opts, algo=None, workspace=None, fill=float("nan")):
    dev = torch.device("cuda", 0)
    dw = torch.full(w_shape, fill, dtype=torch.float32, device=dev)
    sg.conv2d_bwd_weight_into(dw, x.to(dev), dy.to(dev), **opts, algo=algo, workspace=workspace)
    torch.cuda.synchronize()
    return dw.cpu().numpy()


GEOMS = [
    ("3x3_pad1", dict(n=2, h=14, w=14, c=64, k=64, r=3, s=3, pad=1)),
    ("3x3_c128_k128", dict(n=2, h=10, w=12, c=128, k=128, r=3, s=3, pad=1)),
    ("stride2_ragged_l", dict(n=3, h=15, w=13, c=64, k=96, r=3, s=3, stride=2, pad=1)),
    ("dil2_asym", dict(n=2, h=12, w=11, c=128, k=64, r=3, s=2, pad=(2, 1), dil=(2, 1))),
    ("k72_ragged_rows", dict(n=2, h=9, w=9, c=64, k=72, r=3, s=3, pad=1)),
    ("c192_ragged_cols", dict(n=1, h=8, w=8, c=192, k=64, r=3, s=3, pad=1)),
    ("1x1_s2", dict(n=2, h=16, w=16, c=256, k=128, r=1, s=1, stride=2)),
    ("7x7_s2_k256", dict(n=1, h=20, w=20, c=64, k=256, r=7, s=7, stride=2, pad=3)),
    ("one_pixel", dict(n=1, h=3, w=3, c=64, k=8, r=3, s=3)),
]


@pytest.mark.parametrize("bn", [0, 64, 128, 256])
@pytest.mark.parametrize("geom", GEOMS, ids=[g[0] for g in GEOMS])
def test_wgrad_geometries(sg, geom, bn):
    name, kw = geom
    kw = dict(kw)
    x, dy, wsh, opts, L = _case(kw.pop("n"), kw.pop("h"), kw.pop("w"), kw.pop("c"), kw.pop("k"), kw.pop("r"),
                                kw.pop("s"), seed=zlib.crc32(name.encode()) % 1000, **kw)
    got = _gpu(sg, x, dy, wsh, opts, algo=make_algo(sg, block_n=bn, wait_limit_ns=WAIT))
    assert sg.last_launch_count() == 1
    ref = ow.conv2d_wgrad(x, dy, wsh, **opts)
    check_close(got, ref, L, 1, 1, f"wgrad {name} bn={bn}")


@pytest.mark.parametrize("forced", [dict(splits=1), dict(splits=3), dict(splits=8), dict(grid=5), dict(grid=37),
                                    dict(splits=4, reduction=1), dict(grid=23, reduction=1),
                                    dict(grid=23, reduction=2)],
                         ids=["splits1", "splits3", "splits8", "grid5", "grid37", "splits4_ordered",
                              "grid23_ordered", "grid23_concurrent"])
def test_wgrad_forced_plans(sg, forced):
    x, dy, wsh, opts, L = _case(4, 16, 16, 128, 128, 3, 3, pad=1, seed=3)  # 16 k-blocks of 64 pixels
    params = sg.make_params(x.shape, wsh, **opts)
    ws = torch.zeros(sg.wgrad_workspace_bytes(params), dtype=torch.uint8, device="cuda")
    got = _gpu(sg, x, dy, wsh, opts, algo=make_algo(sg, wait_limit_ns=WAIT, **forced), workspace=ws)
    ref = ow.conv2d_wgrad(x, dy, wsh, **opts)
    check_close(got, ref, L, 1, 1, f"wgrad forced {forced}")
    assert int(torch.count_nonzero(ws)) == 0
    assert sg.status(ws) == 0


@pytest.mark.parametrize("bn", [64, 128, 256])
def test_wgrad_integer_inputs_exact(sg, bn):
    x, dy, wsh, opts, L = _case(2, 11, 13, 128, 128, 3, 3, stride=(1, 2), pad=1, seed=7, ints=True)
    got = _gpu(sg, x, dy, wsh, opts, algo=make_algo(sg, block_n=bn, wait_limit_ns=WAIT))
    ref = ow.conv2d_wgrad(x, dy, wsh, **opts)
    assert np.array_equal(got, ref), f"{int(np.count_nonzero(got != ref))} of {got.size} differ"


def test_wgrad_ordered_reduction_is_reproducible(sg):
    x, dy, wsh, opts, L = _case(4, 14, 14, 64, 64, 3, 3, pad=1, seed=9)
    algo = make_algo(sg, splits=6, reduction=1, wait_limit_ns=WAIT)
    a = _gpu(sg, x, dy, wsh, opts, algo=algo)
    b = _gpu(sg, x, dy, wsh, opts, algo=algo)
    assert np.array_equal(a, b)


def test_wgrad_empty_batch_is_zero(sg):
    dev = torch.device("cuda", 0)
    x = torch.zeros((0, 6, 6, 64), dtype=torch.bfloat16, device=dev)
    dy = torch.zeros((0, 6, 6, 16), dtype=torch.bfloat16, device=dev)
    dw = sg.conv2d_bwd_weight(x, dy, (16, 3, 3, 64), padding=1)
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(dw)) == 0


@pytest.mark.parametrize("shape,groups", [(((1, 6, 6, 32), (16, 3, 3, 32)), 1),   # C % 64 != 0
                                          (((1, 6, 6, 64), (12, 3, 3, 64)), 1),   # K % 8 != 0
                                          (((1, 6, 6, 128), (64, 3, 3, 64)), 2)])  # groups
def test_wgrad_unsupported_shapes_refused(sg, shape, groups):
    xs, ws = shape
    dev = torch.device("cuda", 0)
    x = torch.zeros(xs, dtype=torch.bfloat16, device=dev)
    p = xs[1] - 2
    dy = torch.zeros((xs[0], p, p, ws[0]), dtype=torch.bfloat16, device=dev)
    with pytest.raises(sg.Conv2dError) as e:
        sg.conv2d_bwd_weight(x, dy, ws, groups=groups)
    assert e.value.code == 2


FULL = ["resnet_56x56_c64", "resnet_28x28_c256", "splitk_7x7_c2048", "proj_56_c256_1x1s2", "dil2_64_c128"]


@pytest.mark.parametrize("name", FULL)
def test_wgrad_full_size_workloads(sg, name):
    """The weight gradient of each eligible workload at full size (the heuristic's plan),
    checked on sampled elements against the oracle one by one."""
    wl = workloads.get(name)
    x, w, _ = workloads.make_inputs(wl)
    o = wl.options()
    dy = workloads.make_output_grad(wl)
    L = dy.shape[0] * dy.shape[1] * dy.shape[2]
    got = _gpu(sg, x, dy, tuple(w.shape), dict(stride=o["stride"], padding=o["padding"], dilation=o["dilation"]))
    assert sg.last_launch_count() == 1
    flat = got.reshape(wl.k, -1)
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    kk = np.concatenate([rng.integers(0, wl.k, 3000), [0, wl.k - 1, 0, wl.k - 1]])
    jj = np.concatenate([rng.integers(0, flat.shape[1], 3000), [0, 0, flat.shape[1] - 1, flat.shape[1] - 1]])
    ref, _ = ow.conv2d_wgrad_points_f64(oracle.widen_bf16(x), oracle.widen_bf16(dy), tuple(w.shape), o["stride"],
                                        o["padding"], o["dilation"], kk, jj)
    check_close(flat[kk, jj], ref, L, 1, 1, f"wgrad {name}")
    assert np.all(np.isfinite(flat)), f"{name}: a gradient element was not written"
