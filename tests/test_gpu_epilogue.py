"""Fused epilogue (ReLU after the bias, bf16 output) against the oracle through the C ABI
(needs a GB300).

The oracle gives the exact value u = conv + bias; the kernel's output must lie in the
range that ReLU and the bf16 rounding map [u - B, u + B] to (B the fp32 parity bound),
and equal the oracle's epilogue exactly where that range is one value.  With integer
inputs the fp32 sums are exact and every output must equal the oracle's exactly."""
import zlib

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import epilogue
from tests.parity import check_epilogue, gpu_conv_epi, make_algo

pytestmark = pytest.mark.gpu

WAIT = 200_000_000  # 0.2 s bound on every device-side wait in these tests
MODES = [(True, False), (False, True), (True, True)]  # (relu, bf16 output)
MODE_IDS = ["relu_f32", "bf16", "relu_bf16"]


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import split_gemm_gb300
    split_gemm_gb300.load_library()
    torch.cuda.set_device(0)
    return split_gemm_gb300


def _case(n, h, w, c, k, r, s, stride=1, pad=0, dil=1, groups=1, bias=True, seed=0, dist="normal"):
    def pair(v):
        return v if isinstance(v, tuple) else (v, v)
    (sh, sw), (ph, pw), (dh, dw) = pair(stride), pair(pad), pair(dil)
    wl = workloads.Workload(f"epi{seed}", n, h, w, c, k, r, s, sh, sw, ph, pw, dh, dw,
                            x_dist=dist, w_dist="he" if dist == "normal" else dist,
                            bias=("normal:0.1" if dist == "normal" else dist) if bias else None, seed=seed,
                            groups=groups)
    x, wt, b = workloads.make_inputs(wl)
    return wl, x, wt, b


def _run(sg, wl, x, w, b, relu_on, out_bf16, algo, what):
    got = gpu_conv_epi(sg, x, w, b, wl.options(), relu_on, out_bf16, algo=algo)
    u = oracle.conv2d_fwd(x, w, b, **wl.options())
    exact = check_epilogue(got, u, wl.c // wl.groups, wl.r, wl.s, relu_on, out_bf16, what)
    return got, u, exact


# Geometry x loader: each loader's epilogue path (vector stores for K % 4 == 0, row
# stores otherwise; the row-window kernel's own epilogue).
LOADER_CASES = [
    ("tma_im2col", dict(n=2, h=14, w=14, c=64, k=128, r=3, s=3, pad=1), 1, 0, 0),
    ("tma_im2col_bm256", dict(n=2, h=16, w=16, c=64, k=64, r=3, s=3, pad=1), 1, 256, 64),
    ("tma_im2col_bn256", dict(n=2, h=10, w=10, c=128, k=256, r=3, s=3, pad=1), 1, 128, 256),
    ("cpasync", dict(n=2, h=9, w=11, c=24, k=80, r=3, s=3, pad=1, stride=2), 2, 0, 0),
    ("scalar", dict(n=2, h=9, w=9, c=5, k=48, r=3, s=3, pad=1), 3, 0, 0),
    ("hybrid", dict(n=2, h=12, w=12, c=64, k=64, r=3, s=3, pad=1), 4, 0, 0),
    ("row_window", dict(n=2, h=40, w=40, c=3, k=64, r=7, s=7, pad=3, stride=2), 5, 0, 0),
    ("tma_box", dict(n=2, h=16, w=16, c=128, k=128, r=3, s=3, pad=1), 6, 0, 0),
    ("halo", dict(n=2, h=14, w=14, c=64, k=64, r=3, s=3, pad=1), 7, 0, 0),
    ("row_stores_k30", dict(n=2, h=8, w=8, c=16, k=30, r=3, s=3, pad=1), 0, 0, 0),
    ("row_window_k30", dict(n=1, h=30, w=30, c=3, k=30, r=3, s=3, pad=1), 5, 0, 0),
    ("grouped_tma", dict(n=2, h=10, w=10, c=128, k=128, r=3, s=3, pad=1, groups=2), 1, 0, 0),
    ("grouped_cpasync", dict(n=2, h=9, w=9, c=64, k=64, r=3, s=3, pad=1, groups=8), 2, 0, 0),
]


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("case", LOADER_CASES, ids=[c[0] for c in LOADER_CASES])
def test_fused_epilogue_loaders(sg, case, mode):
    name, geom, loader, bm, bn = case
    kw = dict(geom)
    wl, x, w, b = _case(kw.pop("n"), kw.pop("h"), kw.pop("w"), kw.pop("c"), kw.pop("k"), kw.pop("r"),
                        kw.pop("s"), seed=41, **kw)
    algo = make_algo(sg, loader=loader, block_m=bm, block_n=bn, wait_limit_ns=WAIT)
    got, u, exact = _run(sg, wl, x, w, b, *mode, algo, f"{name} {wl.describe()}")
    assert sg.last_launch_count() == 1
    if mode[0]:
        assert np.all(got >= 0.0)


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("loader", [1, 2, 5])
def test_fused_epilogue_integer_inputs_exact(sg, loader, mode):
    """Integer inputs: fp32 sums are exact, so every output equals the oracle's epilogue."""
    if loader == 5:
        wl, x, w, b = _case(2, 30, 30, 3, 64, 7, 7, stride=2, pad=3, seed=5, dist="int:-3:3")
    else:
        wl, x, w, b = _case(2, 10, 12, 64, 128, 3, 3, pad=1, seed=5, dist="int:-3:3")
    algo = make_algo(sg, loader=loader, wait_limit_ns=WAIT)
    got = gpu_conv_epi(sg, x, w, b, wl.options(), *mode, algo=algo)
    u = oracle.conv2d_fwd(x, w, b, **wl.options())
    want = epilogue.apply(u, *mode)
    assert np.array_equal(got, want), f"{int(np.count_nonzero(got != want))} of {got.size} outputs differ"


def test_fused_long_reduction_splits_through_the_partial_buffer(sg):
    """A small-output, long-reduction problem: the fused call splits every tile like the
    plain path (classic split-K), sums the splits in the workspace's fp32 buffer, and the
    last CTA of each tile finishes it; the workspace is left zero."""
    wl, x, w, b = _case(2, 7, 7, 1024, 128, 3, 3, pad=1, seed=8)
    params = sg.make_params(x.shape, w.shape, **wl.options())
    plain = sg.query_algo(params)
    fused = sg.query_algo(params, relu=True, out_bf16=True)
    assert plain.splits > 1 and fused.splits == plain.splits
    need = sg.epi_workspace_bytes(params, None, True, True)
    assert need >= sg.workspace_bytes(params) + 98 * 128 * 4
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for mode in MODES:
        got = gpu_conv_epi(sg, x, w, b, wl.options(), *mode, algo=make_algo(sg, wait_limit_ns=WAIT), workspace=ws)
        u = oracle.conv2d_fwd(x, w, b, **wl.options())
        check_epilogue(got, u, wl.c, wl.r, wl.s, *mode, f"long reduction {mode}")
        assert int(torch.count_nonzero(ws)) == 0
        assert sg.status(ws) == 0


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("forced", [dict(splits=2), dict(splits=5, block_n=64), dict(grid=3, block_n=128),
                                    dict(grid=7, block_n=64, loader=2), dict(splits=3, block_m=256, block_n=64),
                                    dict(splits=4, loader=3), dict(splits=1), dict(grid=1, block_n=128)],
                         ids=["splits2", "splits5_bn64", "streamk3", "streamk7_cpasync", "splits3_bm256",
                              "splits4_scalar_k62", "splits1", "grid1"])
def test_fused_forced_plans(sg, forced, mode):
    """Forced splits and stream-K grids, most of them cutting tiles: vector stores (K = 128)
    and row stores (K = 62 with the scalar loader); splits=1 and grid=1 cut nothing."""
    k = 62 if forced.get("loader") == 3 else 128
    wl, x, w, b = _case(1, 7, 7, 512 if forced.get("loader") != 3 else 40, k, 3, 3, pad=1, seed=9)
    algo = make_algo(sg, wait_limit_ns=WAIT, **forced)
    params = sg.make_params(x.shape, w.shape, **wl.options())
    need = sg.epi_workspace_bytes(params, algo, *mode)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    got = gpu_conv_epi(sg, x, w, b, wl.options(), *mode, algo=algo, workspace=ws)
    u = oracle.conv2d_fwd(x, w, b, **wl.options())
    check_epilogue(got, u, wl.c, wl.r, wl.s, *mode, f"forced {forced}")
    assert int(torch.count_nonzero(ws)) == 0, "the partial-sum buffer or a counter was left non-zero"
    assert sg.status(ws) == 0
    if need > sg.workspace_bytes(params):
        # Without room for the partial-sum buffer the call is refused before any launch.
        small = torch.zeros(sg.workspace_bytes(params), dtype=torch.uint8, device="cuda")
        with pytest.raises(sg.Conv2dError) as ei:
            gpu_conv_epi(sg, x, w, b, wl.options(), *mode, algo=algo, workspace=small)
        assert ei.value.code == 4
    else:
        assert forced in (dict(splits=1), dict(grid=1, block_n=128))


@pytest.mark.parametrize("relu_on", [False, True])
@pytest.mark.parametrize("case", LOADER_CASES, ids=[c[0] for c in LOADER_CASES])
def test_fused_bf16_matches_rounded_fp32_path(sg, case, relu_on):
    """Same plan (whole tiles), same accumulation order: the bf16 output is the plain fp32
    output put through ReLU and round-to-nearest-even (the oracle's rounding, applied to the
    kernel's own fp32 values), bit for bit.  The fp32 parity bound is wide next to the bf16
    spacing, so this is the check that pins the conversion itself on every element."""
    name, geom, loader, bm, bn = case
    kw = dict(geom)
    wl, x, w, b = _case(kw.pop("n"), kw.pop("h"), kw.pop("w"), kw.pop("c"), kw.pop("k"), kw.pop("r"),
                        kw.pop("s"), seed=12, **kw)
    algo = make_algo(sg, loader=loader, block_m=bm, block_n=bn, splits=1, wait_limit_ns=WAIT)
    plain = gpu_conv_epi(sg, x, w, b, wl.options(), False, False, algo=algo)
    fused = gpu_conv_epi(sg, x, w, b, wl.options(), relu_on, True, algo=algo)
    want = epilogue.round_bf16(np.maximum(plain, 0.0) if relu_on else plain)
    assert np.array_equal(fused, want), f"{name}: {int(np.count_nonzero(fused != want))} of {fused.size} differ"
    relu_f32 = gpu_conv_epi(sg, x, w, b, wl.options(), True, False, algo=algo) if relu_on else None
    if relu_on:
        assert np.array_equal(relu_f32, np.maximum(plain, 0.0))


def test_fused_empty_batch(sg):
    wl, x, w, b = _case(1, 6, 6, 16, 16, 3, 3, pad=1, seed=1)
    x0 = x[:0]
    got = gpu_conv_epi(sg, x0, w, b, wl.options(), True, True)
    assert got.shape == (0, 6, 6, 16)


def _sample_points(p_total, k, count, seed):
    rng = np.random.default_rng(seed)
    m = np.concatenate([rng.integers(0, p_total, count), [0, p_total - 1] * 4])
    kk = np.concatenate([rng.integers(0, k, count), [0, k - 1, 0, k - 1, k // 2, k // 2, 1 % k, k - 2 if k > 1 else 0]])
    return m, kk


FULL = list(workloads.ORDER) + list(workloads.GROUPED)


@pytest.mark.parametrize("name", FULL)
def test_fused_full_size_workloads(sg, name):
    """Each workload at full size with ReLU and a bf16 output (the heuristic's fused plan),
    checked on sampled outputs against the oracle one by one."""
    wl = workloads.get(name)
    x, w, b = workloads.make_inputs(wl)
    got = gpu_conv_epi(sg, x, w, b, wl.options(), True, True, algo=make_algo(sg, wait_limit_ns=WAIT))
    params = sg.make_params(x.shape, w.shape, **wl.options())
    # One launch, or two for block-diagonal grouped tiles (the weight expansion first).
    assert sg.last_launch_count() == (2 if sg.query_algo(params).loader == sg.LOADER_BLOCKDIAG else 1)
    n, p, q, k = got.shape
    flat = got.reshape(n * p * q, k)
    m_idx, k_idx = _sample_points(n * p * q, k, 6000, seed=zlib.crc32(name.encode()))
    u = oracle.conv2d_fwd_points(x, w, b, *(wl.options()[key] for key in ("stride", "padding", "dilation")),
                                 m_idx, k_idx, groups=wl.groups)
    check_epilogue(flat[m_idx, k_idx], u, wl.c // wl.groups, wl.r, wl.s, True, True, name)
    assert np.all(np.isfinite(flat)), f"{name}: an output element was not written"
