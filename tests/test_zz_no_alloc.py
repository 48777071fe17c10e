"""The no-allocation entry point, for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (a plugin whose host framework owns all
device memory and offers no workspace hook, a deployment that forbids
allocation after start-up, a latency-critical loop that must not risk the
device-wide synchronisation an allocation can cause), so they cannot hand
conv2d_fwd a workspace.  conv2d_fwd_noalloc uses a static scratch array inside
the library instead.  These tests call it through the C ABI and compare its
output with conv2d_fwd's (own workspace), within the parity tolerance, on two
calls in a row; the second call also checks that the scratch left behind by
the first does not leak into the result.  This file is collected last on
purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import check_close

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 65536  # CONV2D_NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import split_gemm_gb300
    split_gemm_gb300.load_library()
    torch.cuda.set_device(0)
    return split_gemm_gb300


def _long_reduction():
    # One output tile, 36 k-blocks: the heuristic splits the reduction, so the
    # split-K semaphores in the scratch array are exercised.
    return workloads.Workload("noalloc_longk", 2, 6, 6, 256, 96, 3, 3, 1, 1, 1, 1, 1, 1,
                              x_dist="uniform", w_dist="uniform", bias="normal:0.1", seed=11)


@pytest.mark.parametrize("wl", [_long_reduction(), workloads.get("splitk_7x7_c2048"),
                                workloads.get("resnet_56x56_c64")], ids=lambda w: w.name)
def test_noalloc_matches_regular_entry_point_twice(sg, wl):
    lib = sg.load_library()
    dev = torch.device("cuda", 0)
    x, w, b = workloads.make_inputs(wl)
    xd, wd = x.to(dev), w.to(dev)
    bd = None if b is None else b.to(dev)
    params = sg.make_params(x.shape, w.shape, **wl.options())
    assert sg.workspace_bytes(params) <= SCRATCH_LIMIT
    p, q = sg.output_shape(params)
    stream = torch.cuda.current_stream(dev).cuda_stream

    ref = sg.conv2d_fwd(xd, wd, bd, **wl.options())  # regular entry point, torch-allocated workspace
    torch.cuda.synchronize()
    ref = ref.cpu().numpy()

    outs = []
    for _ in range(2):
        y = torch.full((wl.n, p, q, wl.k), float("nan"), dtype=torch.float32, device=dev)
        rc = lib.conv2d_fwd_noalloc(ctypes.byref(params), xd.data_ptr(), wd.data_ptr(),
                                    None if bd is None else bd.data_ptr(), y.data_ptr(), stream)
        assert rc == 0, sg.strerror(rc)
        torch.cuda.synchronize()
        outs.append(y.cpu().numpy())
    for got in outs:
        check_close(got, ref.astype(np.float64), wl.c, wl.r, wl.s, f"{wl.name} noalloc vs conv2d_fwd")
    if wl.name == "noalloc_longk":  # small enough to also hold against the oracle here
        check_close(outs[1], oracle.conv2d_fwd(x, w, b, **wl.options()), wl.c, wl.r, wl.s, "noalloc vs oracle")


def test_noalloc_rejects_problems_beyond_the_scratch_size(sg):
    lib = sg.load_library()
    # 40 x 230 x 230 pixels, 64 channels: 16532 tiles of 128 x 64, more semaphores
    # than the 64 KiB array holds.  Rejected on the host before anything is enqueued.
    params = sg.make_params((40, 230, 230, 8), (64, 1, 1, 8))
    assert sg.workspace_bytes(params) > SCRATCH_LIMIT
    dummy = torch.zeros(64, dtype=torch.float32, device="cuda")
    rc = lib.conv2d_fwd_noalloc(ctypes.byref(params), dummy.data_ptr(), dummy.data_ptr(), None,
                                dummy.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 7  # CONV2D_ERR_SCRATCH_LIMIT
    assert "static scratch" in sg.strerror(rc)
