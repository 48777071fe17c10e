"""The CTA-pair kernel (256-pixel tiles on clusters of two CTAs, 2-CTA tensor-core MMAs)
against the oracle, element by element through the C ABI (needs a GB300)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import check_close, check_epilogue, gpu_conv, gpu_conv_epi, make_algo

pytestmark = pytest.mark.gpu

WAIT = 200_000_000  # 0.2 s bound on every device-side wait in these tests
PAIR = 9            # CONV2D_LOADER_TMA_PAIR
KB = {1: 2, 2: 4}   # CONV2D_DEBUG_PAIR_KB1 / KB2: one or two k-blocks per pipeline stage


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import split_gemm_gb300
    split_gemm_gb300.load_library()
    torch.cuda.set_device(0)
    return split_gemm_gb300


def _case(n, h, w, c, k, r, s, stride=1, pad=0, dil=1, bias=True, seed=0, dist="normal"):
    def two(v):
        return v if isinstance(v, tuple) else (v, v)
    (sh, sw), (ph, pw), (dh, dw) = two(stride), two(pad), two(dil)
    wl = workloads.Workload(f"pair{seed}", n, h, w, c, k, r, s, sh, sw, ph, pw, dh, dw,
                            x_dist=dist, w_dist="he" if dist == "normal" else dist,
                            bias=("normal:0.1" if dist == "normal" else dist) if bias else None, seed=seed)
    x, wt, b = workloads.make_inputs(wl)
    return wl, x, wt, b


def _check(sg, wl, x, w, b, algo, what):
    got = gpu_conv(sg, x, w, b, wl.options(), algo=algo)
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    check_close(got, ref, wl.c, wl.r, wl.s, what)
    return got, ref


# Shapes chosen to hit every edge of the pair tiling: M below one 256-pixel tile (the peer CTA's
# half partly or wholly past the output), ragged M and K, an odd number of 64-wide k-blocks
# (the last stage holds one), strides, dilation, asymmetric windows, 1x1, 5x5.
GEOMETRIES = {
    "m200_k80_3x3": (2, 10, 10, 64, 80, 3, 3, 1, 1, 1),
    "m588_k136_3x3": (3, 14, 14, 128, 136, 3, 3, 1, 1, 1),
    "m84_s2_k256": (2, 13, 11, 64, 256, 3, 3, 2, 1, 1),
    "m400_dil2_k64": (1, 20, 20, 128, 64, 3, 3, 1, 2, 2),
    "1x1_c192_k320": (4, 9, 9, 192, 320, 1, 1, 1, 0, 1),
    "asym_3x2_k48": (2, 8, 12, 64, 48, 3, 2, (2, 1), (1, 0), 1),
    "5x5_c256_k128": (1, 16, 16, 256, 128, 5, 5, 1, 2, 1),
    "m40_k16": (1, 5, 8, 64, 16, 3, 3, 1, 1, 1),
}


@pytest.mark.parametrize("kb", [1, 2])
@pytest.mark.parametrize("bn", [64, 128, 256])
@pytest.mark.parametrize("name", sorted(GEOMETRIES))
def test_pair_geometries_each_width(sg, name, bn, kb):
    n, h, w_, c, k, r, s, stride, pad, dil = GEOMETRIES[name]
    wl, x, w, b = _case(n, h, w_, c, k, r, s, stride, pad, dil, seed=sum(map(ord, name)) % 1000)
    algo = make_algo(sg, loader=PAIR, block_n=bn, wait_limit_ns=WAIT, debug_flags=KB[kb])
    _check(sg, wl, x, w, b, algo, f"{name} bn={bn} kb={kb}")


@pytest.mark.parametrize("split", [0, 3])
@pytest.mark.parametrize("bn", [64, 256])
@pytest.mark.parametrize("name", sorted(GEOMETRIES))
def test_pair_tma_store_path(sg, name, bn, split):
    """The TMA store path (a measurement hook): whole tiles and, with three splits, TMA stores
    of split 0 and TMA reductions of the later splits (rows past a span added as zeros)."""
    n, h, w_, c, k, r, s, stride, pad, dil = GEOMETRIES[name]
    wl, x, w, b = _case(n, h, w_, c, k, r, s, stride, pad, dil, seed=sum(map(ord, name)) % 997)
    algo = make_algo(sg, loader=PAIR, block_n=bn, wait_limit_ns=WAIT, debug_flags=sg.DEBUG_TMA_STORE,
                     splits=split)
    try:
        _check(sg, wl, x, w, b, algo, f"{name} bn={bn} splits={split} TMA stores")
    except sg.Conv2dError as e:  # more splits than stages
        assert split and e.code == 2


@pytest.mark.parametrize("name", ["m588_k136_3x3", "1x1_c192_k320", "m200_k80_3x3", "asym_3x2_k48"])
def test_pair_integer_inputs_exact(sg, name):
    """Small integers: every product and partial sum is exact in fp32, so the result must equal
    the oracle's bit for bit whatever the summation order."""
    n, h, w_, c, k, r, s, stride, pad, dil = GEOMETRIES[name]
    wl, x, w, b = _case(n, h, w_, c, k, r, s, stride, pad, dil, seed=3, dist="int:-3:3")
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=PAIR, wait_limit_ns=WAIT))
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    assert np.array_equal(got.astype(np.float64), ref)


@pytest.fixture(scope="module")
def long_k():
    # M = 2*14*14 = 392 pixels (two pair tiles, the second with 136 valid rows: one full half and
    # one partly valid), K = 192, C*R*S = 256*9 = 2304 (36 k-blocks, 18 stages).
    wl, x, w, b = _case(2, 14, 14, 256, 192, 3, 3, 1, 1, 1, seed=11, dist="uniform")
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    return wl, x, w, b, ref


@pytest.mark.parametrize("kb", [1, 2])
@pytest.mark.parametrize("reduction", [1, 2])
@pytest.mark.parametrize("split", [("splits", 2), ("splits", 5), ("splits", 18), ("grid", 3), ("grid", 7), ("grid", 31)])
def test_pair_cut_tiles_both_reductions(sg, long_k, split, reduction, kb):
    wl, x, w, b, ref = long_k
    dev = torch.device("cuda", 0)
    params = sg.make_params(x.shape, w.shape, **wl.options())
    ws = torch.zeros(sg.workspace_bytes(params), dtype=torch.uint8, device=dev)
    algo = make_algo(sg, loader=PAIR, wait_limit_ns=WAIT, reduction=reduction, debug_flags=KB[kb],
                     **{split[0]: split[1]})
    got = gpu_conv(sg, x, w, b, wl.options(), algo=algo, workspace=ws)
    check_close(got, ref, wl.c, wl.r, wl.s, f"pair {split} reduction {reduction}")
    assert int(torch.count_nonzero(ws)) == 0  # semaphores back at zero
    assert sg.status(ws) == 0


def test_pair_ordered_reduction_reproducible(sg, long_k):
    wl, x, w, b, _ = long_k
    algo = make_algo(sg, loader=PAIR, grid=7, reduction=1, wait_limit_ns=WAIT)
    first = gpu_conv(sg, x, w, b, wl.options(), algo=algo)
    again = gpu_conv(sg, x, w, b, wl.options(), algo=algo)
    assert np.array_equal(first, again)


def test_pair_output_prior_contents_ignored(sg, long_k):
    wl, x, w, b, ref = long_k
    dev = torch.device("cuda", 0)
    y = torch.full((2, 14, 14, 192), 1e30, dtype=torch.float32, device=dev)
    sg.conv2d_fwd_into(y, x.to(dev), w.to(dev), b.to(dev), **wl.options(),
                       algo=make_algo(sg, loader=PAIR, splits=4, wait_limit_ns=WAIT))
    torch.cuda.synchronize()
    check_close(y.cpu().numpy(), ref, wl.c, wl.r, wl.s, "poisoned output")


@pytest.mark.parametrize("kb", [1, 2])
@pytest.mark.parametrize("reduction", [1, 2])
def test_pair_bounded_wait_reports_timeout_and_recovers(sg, long_k, reduction, kb):
    """Split 0 never signals (test hook): the later splits' waits run out after 20 ms, the
    status word reports a timeout, and the next call on the same workspace is correct."""
    wl, x, w, b, ref = long_k
    dev = torch.device("cuda", 0)
    params = sg.make_params(x.shape, w.shape, **wl.options())
    ws = torch.zeros(sg.workspace_bytes(params), dtype=torch.uint8, device=dev)
    hook = make_algo(sg, loader=PAIR, splits=3, debug_flags=sg.DEBUG_SKIP_SIGNAL | KB[kb], wait_limit_ns=20_000_000,
                     reduction=reduction)
    gpu_conv(sg, x, w, b, wl.options(), algo=hook, workspace=ws)
    assert sg.status(ws) == 6  # CONV2D_ERR_TIMEOUT
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=PAIR, splits=3, wait_limit_ns=WAIT),
                   workspace=ws)
    check_close(got, ref, wl.c, wl.r, wl.s, "after timeout")
    assert sg.status(ws) == 0


@pytest.mark.parametrize("mode", [(True, False), (False, True), (True, True)])
@pytest.mark.parametrize("name", ["m588_k136_3x3", "m200_k80_3x3", "1x1_c192_k320"])
def test_pair_fused_epilogue_whole_tiles(sg, name, mode):
    n, h, w_, c, k, r, s, stride, pad, dil = GEOMETRIES[name]
    wl, x, w, b = _case(n, h, w_, c, k, r, s, stride, pad, dil, seed=5)
    got = gpu_conv_epi(sg, x, w, b, wl.options(), *mode, algo=make_algo(sg, loader=PAIR, wait_limit_ns=WAIT))
    u = oracle.conv2d_fwd(x, w, b, **wl.options())
    check_epilogue(got.astype(np.float64), u, wl.c, wl.r, wl.s, *mode, f"{name} fused {mode}")


def test_pair_fused_epilogue_refuses_cut_tiles(sg, long_k):
    wl, x, w, b, _ = long_k
    with pytest.raises(sg.Conv2dError) as e:
        gpu_conv_epi(sg, x, w, b, wl.options(), True, True, algo=make_algo(sg, loader=PAIR, splits=2))
    assert e.value.code == 2  # CONV2D_ERR_UNSUPPORTED


GROUPED = {
    "g2_cg64_kg64": (2, 10, 10, 128, 128, 3, 3, 1, 1, 1, 2),
    "g4_cg64_kg128_s2": (2, 13, 11, 256, 512, 3, 3, 2, 1, 1, 4),
    "g2_cg128_kg96": (1, 9, 12, 256, 192, 3, 3, 1, 1, 2, 2),
    "g8_cg64_kg64_1x1": (3, 8, 8, 512, 512, 1, 1, 1, 0, 1, 8),
}


@pytest.mark.parametrize("split", [0, 3])
@pytest.mark.parametrize("name", sorted(GROUPED))
def test_pair_grouped(sg, name, split):
    """Groups of 64+ channels on the pair kernel: column blocks never straddle a group, each
    group's im2col boxes start at its first input channel; whole and cut tiles."""
    n, h, w_, c, k, r, s, stride, pad, dil, groups = GROUPED[name]
    wl = workloads.Workload(f"pg{groups}", n, h, w_, c, k, r, s, stride, stride, pad, pad, dil, dil,
                            x_dist="normal", w_dist="he", bias="normal:0.1", seed=sum(map(ord, name)) % 1000,
                            groups=groups)
    x, w, b = workloads.make_inputs(wl)
    algo = make_algo(sg, loader=PAIR, wait_limit_ns=WAIT, splits=split)
    stages = -(-(c // groups * r * s // 64) // 2)
    if split > stages:  # every split needs a stage
        with pytest.raises(sg.Conv2dError) as e:
            gpu_conv(sg, x, w, b, wl.options(), algo=algo)
        assert e.value.code == 2
        return
    got = gpu_conv(sg, x, w, b, wl.options(), algo=algo)
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    check_close(got, ref, c // groups, r, s, f"pair grouped {name} splits={split}")


def test_pair_grouped_integer_exact(sg):
    wl = workloads.Workload("pgi", 2, 9, 10, 256, 256, 3, 3, 1, 1, 1, 1, 1, 1, x_dist="int:-3:3", w_dist="int:-3:3",
                            bias="int:-3:3", seed=5, groups=4)
    x, w, b = workloads.make_inputs(wl)
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=PAIR, wait_limit_ns=WAIT))
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    assert np.array_equal(got.astype(np.float64), ref)


@pytest.mark.parametrize("shape", [
    (1, 8, 8, 64, 64, 3, 3, 1, 1, 1, 2),    # groups of 32 channels
    (1, 8, 8, 32, 64, 3, 3, 1, 1, 1, 1),    # C % 64 != 0
    (1, 8, 8, 64, 66, 3, 3, 1, 1, 1, 1),    # K % 4 != 0
])
def test_pair_refuses_ineligible_shapes(sg, shape):
    n, h, w_, c, k, r, s, stride, pad, dil, groups = shape
    dev = torch.device("cuda", 0)
    x = torch.zeros((n, h, w_, c), dtype=torch.bfloat16, device=dev)
    w = torch.zeros((k, r, s, c // groups), dtype=torch.bfloat16, device=dev)
    with pytest.raises(sg.Conv2dError) as e:
        sg.conv2d_fwd(x, w, None, stride, pad, dil, groups, algo=make_algo(sg, loader=PAIR))
    assert e.value.code == 2


@pytest.mark.parametrize("kb", [1, 2])
@pytest.mark.parametrize("name", ["resnet_56x56_c64", "resnet_28x28_c256", "splitk_7x7_c2048",
                                  "proj_56_c256_1x1s2", "dil2_64_c128"])
def test_pair_full_size_workloads(sg, name, kb):
    wl = workloads.get(name)
    x, w, b = workloads.make_inputs(wl)
    algo = make_algo(sg, loader=PAIR, wait_limit_ns=WAIT, debug_flags=KB[kb])
    got, ref = _check(sg, wl, x, w, b, algo, name + " pair")
    assert sg.last_launch_count() == 1
