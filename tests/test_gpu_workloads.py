"""Every benchmark workload at full size, in the launch configuration the benchmark times,
against the oracle on every output element (needs a GB300)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import check_close, gpu_conv, make_algo

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import split_gemm_gb300
    split_gemm_gb300.load_library()
    torch.cuda.set_device(0)
    return split_gemm_gb300


@pytest.mark.parametrize("name", workloads.ORDER)
def test_workload_full_parity(sg, name):
    wl = workloads.get(name)
    x, w, b = workloads.make_inputs(wl)
    got = gpu_conv(sg, x, w, b, wl.options())
    assert sg.last_launch_count() == 1
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    check_close(got, ref, wl.c, wl.r, wl.s, name)
    # The heuristic's configuration with the ordered reduction is bitwise reproducible.
    ordered = make_algo(sg, reduction=sg.REDUCTION_ORDERED)
    first = gpu_conv(sg, x, w, b, wl.options(), algo=ordered)
    again = gpu_conv(sg, x, w, b, wl.options(), algo=ordered)
    assert np.array_equal(first, again)
    check_close(first, ref, wl.c, wl.r, wl.s, name + " ordered")


@pytest.mark.parametrize("name", ["resnet_56x56_c64", "splitk_7x7_c2048"])
def test_host_entry_point_matches_device_entry_point(sg, name):
    wl = workloads.get(name)
    x, w, b = workloads.make_inputs(wl)
    params = sg.make_params(x.shape, w.shape, **wl.options())
    p, q = sg.output_shape(params)
    staging = torch.zeros(sg.host_staging_bytes(params), dtype=torch.uint8, device="cuda")
    xh, wh = x.pin_memory(), w.pin_memory()
    bh = None if b is None else b.pin_memory()
    yh = torch.empty((wl.n, p, q, wl.k), dtype=torch.float32).pin_memory()
    sg.conv2d_fwd_host(xh, wh, bh, yh, params, staging)
    torch.cuda.synchronize()
    dev = gpu_conv(sg, x, w, b, wl.options())
    # Same configuration; a split reduction that adds concurrently may round differently.
    check_close(yh.numpy(), dev.astype(np.float64), wl.c, wl.r, wl.s, name + " host vs device")
