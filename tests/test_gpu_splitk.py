"""Split-K with the serialised in-place reduction, and the bounded-wait failure path (needs a GB300)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import check_close, gpu_conv, make_algo

pytestmark = pytest.mark.gpu

WAIT = 200_000_000


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import split_gemm_gb300
    split_gemm_gb300.load_library()
    torch.cuda.set_device(0)
    return split_gemm_gb300


@pytest.fixture(scope="module")
def long_k_case():
    # M = 2*6*6 = 72 pixels, K = 96 channels, C*R*S = 256*9 = 2304 (36 k-blocks).
    wl = workloads.Workload("longk", 2, 6, 6, 256, 96, 3, 3, 1, 1, 1, 1, 1, 1,
                            x_dist="uniform", w_dist="uniform", bias="normal:0.1", seed=7)
    x, w, b = workloads.make_inputs(wl)
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    return wl, x, w, b, ref


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 36])
@pytest.mark.parametrize("loader", [1, 2, 4])
def test_forced_splits_match_oracle(sg, long_k_case, splits, loader):
    wl, x, w, b, ref = long_k_case
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, splits=splits, loader=loader, wait_limit_ns=WAIT))
    check_close(got, ref, wl.c, wl.r, wl.s, f"splits={splits} loader={loader}")


@pytest.mark.parametrize("splits", [2, 5])
def test_forced_splits_256_pixel_tiles(sg, long_k_case, splits):
    wl, x, w, b, ref = long_k_case
    got = gpu_conv(sg, x, w, b, wl.options(),
                   algo=make_algo(sg, splits=splits, loader=1, block_m=256, wait_limit_ns=WAIT))
    check_close(got, ref, wl.c, wl.r, wl.s, f"BM=256 splits={splits}")


def test_splits_agree_and_are_deterministic(sg, long_k_case):
    wl, x, w, b, _ = long_k_case
    outs = {}
    for s in (1, 5):
        algo = make_algo(sg, splits=s, wait_limit_ns=WAIT, reduction=sg.REDUCTION_ORDERED)
        a = gpu_conv(sg, x, w, b, wl.options(), algo=algo)
        c = gpu_conv(sg, x, w, b, wl.options(), algo=algo)
        assert np.array_equal(a, c), f"splits={s} is not bitwise reproducible"
        outs[s] = a
    # Different split factors sum in different orders: equal within the parity bound.
    check_close(outs[5], outs[1].astype(np.float64), wl.c, wl.r, wl.s, "splits 5 vs 1")


@pytest.mark.parametrize("reduction", [1, 2])
@pytest.mark.parametrize("splits", [2, 6, 36])
def test_reduction_modes_match_oracle(sg, long_k_case, reduction, splits):
    wl, x, w, b, ref = long_k_case
    algo = make_algo(sg, splits=splits, wait_limit_ns=WAIT, reduction=reduction)
    got = gpu_conv(sg, x, w, b, wl.options(), algo=algo)
    check_close(got, ref, wl.c, wl.r, wl.s, f"splits={splits} reduction={reduction}")


@pytest.mark.parametrize("grid", [5, 13, 30])
def test_concurrent_reduction_stream_k(sg, long_k_case, grid):
    # Stream-K ranges cut the tiles at uneven points; one CTA may hold the tail of
    # one tile and the head of the next.
    wl, x, w, b, ref = long_k_case
    algo = make_algo(sg, grid=grid, wait_limit_ns=WAIT, reduction=sg.REDUCTION_CONCURRENT)
    got = gpu_conv(sg, x, w, b, wl.options(), algo=algo)
    check_close(got, ref, wl.c, wl.r, wl.s, f"grid={grid} concurrent")


def test_concurrent_reduction_row_stores(sg):
    # K % 4 != 0: the row-per-thread epilogue adds with scalar atomics.
    wl = workloads.Workload("longk_odd", 2, 6, 6, 256, 30, 3, 3, 1, 1, 1, 1, 1, 1,
                            x_dist="uniform", w_dist="uniform", bias="normal:0.1", seed=9)
    x, w, b = workloads.make_inputs(wl)
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    got = gpu_conv(sg, x, w, b, wl.options(),
                   algo=make_algo(sg, splits=4, wait_limit_ns=WAIT, reduction=sg.REDUCTION_CONCURRENT))
    check_close(got, ref, wl.c, wl.r, wl.s, "K=30 splits=4 concurrent")


@pytest.mark.parametrize("reduction", [1, 2])
def test_workspace_left_zeroed_both_modes(sg, long_k_case, reduction):
    wl, x, w, b, _ = long_k_case
    dev = torch.device("cuda", 0)
    params = sg.make_params(x.shape, w.shape, **wl.options())
    ws = torch.zeros(sg.workspace_bytes(params), dtype=torch.uint8, device=dev)
    for algo in (make_algo(sg, splits=5, wait_limit_ns=WAIT, reduction=reduction),
                 make_algo(sg, grid=11, wait_limit_ns=WAIT, reduction=reduction)):
        gpu_conv(sg, x, w, b, wl.options(), algo=algo, workspace=ws)
        assert int(torch.count_nonzero(ws)) == 0
    assert sg.status(ws) == 0


def test_output_prior_contents_ignored_under_split(sg, long_k_case):
    wl, x, w, b, ref = long_k_case
    dev = torch.device("cuda", 0)
    xd, wd, bd = x.to(dev), w.to(dev), b.to(dev)
    y = torch.full((2, 6, 6, 96), 1e30, dtype=torch.float32, device=dev)
    sg.conv2d_fwd_into(y, xd, wd, bd, **wl.options(), algo=make_algo(sg, splits=4, wait_limit_ns=WAIT))
    torch.cuda.synchronize()
    check_close(y.cpu().numpy(), ref, wl.c, wl.r, wl.s, "poisoned output")


def test_workspace_left_zeroed(sg, long_k_case):
    wl, x, w, b, _ = long_k_case
    dev = torch.device("cuda", 0)
    params = sg.make_params(x.shape, w.shape, **wl.options())
    ws = torch.zeros(sg.workspace_bytes(params), dtype=torch.uint8, device=dev)
    gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, splits=6, wait_limit_ns=WAIT), workspace=ws)
    assert int(torch.count_nonzero(ws)) == 0
    assert sg.status(ws) == 0


def test_split_without_workspace_is_an_error(sg, long_k_case):
    wl, x, w, b, _ = long_k_case
    dev = torch.device("cuda", 0)
    tiny = torch.zeros(16, dtype=torch.uint8, device=dev)
    with pytest.raises(sg.Conv2dError) as e:
        gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, splits=2), workspace=tiny)
    assert e.value.code == 4


@pytest.mark.parametrize("reduction", [1, 2])
def test_bounded_wait_reports_timeout_and_recovers(sg, long_k_case, reduction):
    """Split 0 never signals (test hook): the later splits' waits run out after
    20 ms, the status word reports a timeout, the context stays usable and the
    reset workspace serves the next call."""
    wl, x, w, b, ref = long_k_case
    dev = torch.device("cuda", 0)
    params = sg.make_params(x.shape, w.shape, **wl.options())
    ws = torch.zeros(sg.workspace_bytes(params), dtype=torch.uint8, device=dev)
    hook = make_algo(sg, splits=3, debug_flags=sg.DEBUG_SKIP_SIGNAL, wait_limit_ns=20_000_000, reduction=reduction)
    gpu_conv(sg, x, w, b, wl.options(), algo=hook, workspace=ws)
    assert sg.status(ws) == 6  # CONV2D_ERR_TIMEOUT
    assert int(torch.count_nonzero(ws)) == 0  # reset by the status call
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, splits=3, wait_limit_ns=WAIT), workspace=ws)
    check_close(got, ref, wl.c, wl.r, wl.s, "after timeout")
    assert sg.status(ws) == 0
