"""Row-window loader (few input channels) vs the CPU oracle (needs a GB300).

The loader pads each pixel to Cp = 8 / stride_w channels and lets the MMA read
overlapping 16-byte-pitch windows of staged input rows, so the cases below walk
every Cp (stride_w 1, 2, 4, 8), C below and at Cp, output rows longer than one
128-pixel tile, row reuse between consecutive output rows (stride_h < R,
dilation_h 1) and its absence, padding on every side, ragged K and K % 4 != 0.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import check_close, gpu_conv, make_algo

pytestmark = pytest.mark.gpu

WAIT = 200_000_000
ROW_WINDOW = 5


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import split_gemm_gb300
    split_gemm_gb300.load_library()
    torch.cuda.set_device(0)
    return split_gemm_gb300


def _wl(name, n, h, w, c, k, r, s, sh=1, sw=1, ph=0, pw=0, dh=1, dist="normal", bias=True, seed=0):
    return workloads.Workload(name, n, h, w, c, k, r, s, sh, sw, ph, pw, dh, 1,
                              x_dist=dist, w_dist="he" if dist == "normal" else dist,
                              bias=("normal:0.1" if dist == "normal" else dist) if bias else None, seed=seed)


CASES = [
    # name, n, h, w, c, k, r, s, sh, sw, ph, pw, dh
    ("stem_like", 2, 40, 40, 3, 64, 7, 7, 2, 2, 3, 3, 1),      # Cp 4, reuse 5 of 7 rows
    ("c3_s1", 1, 9, 9, 3, 20, 3, 3, 1, 1, 1, 1, 1),            # Cp 8, K ragged in N
    ("c3_k130", 1, 9, 9, 3, 130, 3, 3, 1, 1, 1, 1, 1),         # BN 256
    ("c1_k5", 3, 5, 7, 1, 5, 3, 3, 1, 1, 1, 1, 1),             # K % 4 != 0: row-per-thread stores
    ("wide_q", 1, 12, 300, 2, 8, 3, 5, 1, 1, 1, 2, 1),         # Q = 300: three column blocks
    ("sw8", 2, 11, 40, 1, 8, 3, 3, 3, 8, 1, 1, 1),             # Cp 1, stride_h >= R: no reuse
    ("dil_h2", 2, 15, 33, 2, 24, 3, 3, 2, 4, 2, 1, 2),         # dilation_h 2: no reuse
    ("c8_s1", 2, 14, 20, 8, 48, 3, 3, 1, 1, 1, 1, 1),          # C == Cp
    ("tall", 2, 30, 17, 4, 32, 11, 1, 1, 2, 5, 0, 1),          # 11 x 1 filter
    ("one_pixel", 1, 1, 1, 3, 16, 1, 1, 1, 1, 0, 0, 1),        # M = 1
    ("weight_passes", 1, 20, 20, 8, 128, 7, 7, 1, 1, 3, 3, 1), # weight copied in 7 passes, T = 2
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_row_window_matches_oracle(sg, case):
    wl = _wl(*case, seed=11)
    x, w, b = workloads.make_inputs(wl)
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=ROW_WINDOW, wait_limit_ns=WAIT))
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    check_close(got, ref, wl.c, wl.r, wl.s, case[0])


@pytest.mark.parametrize("grid", [1, 2, 7])
def test_row_window_few_ctas(sg, grid):
    # Few CTAs: long tile ranges, many reused rows, the row ring wraps many times.
    wl = _wl("stem_like", 2, 40, 40, 3, 64, 7, 7, 2, 2, 3, 3, seed=5)
    x, w, b = workloads.make_inputs(wl)
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=ROW_WINDOW, grid=grid, wait_limit_ns=WAIT))
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    check_close(got, ref, wl.c, wl.r, wl.s, f"grid={grid}")


@pytest.mark.parametrize("seed", range(4))
def test_row_window_integer_inputs_exact(sg, seed):
    # Small integers: every partial sum is exact in fp32, so the result must be exact.
    wl = _wl("ints", 2, 23, 29, 3, 40, 5, 5, 2, 2, 2, 2, dist="int:-3:3", seed=seed)
    x, w, b = workloads.make_inputs(wl)
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=ROW_WINDOW, wait_limit_ns=WAIT))
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    assert np.array_equal(got.astype(np.float64), ref)


def test_row_window_chosen_for_small_channels(sg):
    wl = workloads.get("stem_224_c3_7x7s2")
    algo = sg.query_algo(sg.make_params((wl.n, wl.h, wl.w, wl.c), (wl.k, wl.r, wl.s, wl.c), **wl.options()))
    assert algo.loader == ROW_WINDOW


@pytest.mark.parametrize("shape", [
    dict(c=16, sw=1, dw=1, k=16),   # C > Cp
    dict(c=3, sw=3, dw=1, k=16),    # stride_w not a power of two
    dict(c=3, sw=1, dw=2, k=16),    # dilation_w 2
    dict(c=3, sw=1, dw=1, k=300),   # more than one tile of channels
])
def test_row_window_rejects_ineligible(sg, shape):
    x = torch.zeros((1, 12, 12, shape["c"]), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((shape["k"], 3, 3, shape["c"]), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sg.Conv2dError) as e:
        sg.conv2d_fwd(x, w, None, stride=(1, shape["sw"]), padding=1, dilation=(1, shape["dw"]),
                      algo=make_algo(sg, loader=ROW_WINDOW))
    assert e.value.code == 2
