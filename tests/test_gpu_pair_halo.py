"""The CTA-pair halo loader (stride 1: whole padded input rows per 64-channel chunk serve every
filter tap; 2-CTA tensor-core MMAs on two images' pixel blocks) against the oracle, element by
element through the C ABI (needs a GB300)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import check_close, check_epilogue, gpu_conv, gpu_conv_epi, make_algo

pytestmark = pytest.mark.gpu

WAIT = 200_000_000  # 0.2 s bound on every device-side wait in these tests
HALO = 10           # CONV2D_LOADER_PAIR_HALO


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import split_gemm_gb300
    split_gemm_gb300.load_library()
    torch.cuda.set_device(0)
    return split_gemm_gb300


def _case(n, h, w, c, k, r, s, pad=0, dil=1, bias=True, seed=0, dist="normal", groups=1):
    def two(v):
        return v if isinstance(v, tuple) else (v, v)
    (ph, pw), (dh, dw) = two(pad), two(dil)
    wl = workloads.Workload(f"halo{seed}", n, h, w, c, k, r, s, 1, 1, ph, pw, dh, dw,
                            x_dist=dist, w_dist="he" if dist == "normal" else dist,
                            bias=("normal:0.1" if dist == "normal" else dist) if bias else None, seed=seed,
                            groups=groups)
    x, wt, b = workloads.make_inputs(wl)
    return wl, x, wt, b


def _check(sg, wl, x, w, b, algo, what):
    got = gpu_conv(sg, x, w, b, wl.options(), algo=algo)
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    check_close(got, ref, wl.c // wl.groups, wl.r, wl.s, what)
    return got, ref


# Edges of the halo tiling: an odd image count (the last pair's second image is absent), a single
# image, 1x1 (one tap: the weight box's second tap reads zeros), 5x5 (an odd tap count), dilation,
# asymmetric windows and pads, no padding, ragged K, a padded row of 202 pixels (a 128-pixel block
# inside one row) and blocks that start mid-row.
GEOMETRIES = {
    "n2_10x10_c64_k80": (2, 10, 10, 64, 80, 3, 3, 1, 1),
    "n3_14x14_c128_k136": (3, 14, 14, 128, 136, 3, 3, 1, 1),
    "n1_20x20_dil2_k64": (1, 20, 20, 128, 64, 3, 3, 2, 2),
    "n4_9x9_1x1_c192_k320": (4, 9, 9, 192, 320, 1, 1, 0, 1),
    "n2_8x12_3x2_pad10_k48": (2, 8, 12, 64, 48, 3, 2, (1, 0), 1),
    "n1_16x16_5x5_c256_k128": (1, 16, 16, 256, 128, 5, 5, 2, 1),
    "n2_12x12_valid_k64": (2, 12, 12, 64, 64, 3, 3, 0, 1),
    "n2_6x200_wide_k64": (2, 6, 200, 64, 64, 3, 3, 1, 1),
    "n5_7x7_c64_k16": (5, 7, 7, 64, 16, 3, 3, 1, 1),
}


SMEM_LIMIT = 232448  # dynamic shared memory one CTA may opt in to


def _halo_smem(wl, bn, taps):
    """Shared memory of the halo kernel: two halo buffers, four stages of `taps` taps of
    bn/2 weight rows, eight 4 KB epilogue slots, barriers and 1 KB alignment slack."""
    wv = wl.w + 2 * wl.pad_w
    max_row = (wv - 1) + (wl.r - 1) * wl.dil_h * wv + (wl.s - 1) * wl.dil_w + 127
    hr = max_row // wv + 1
    halo = (hr * wv * 128 + 1023) // 1024 * 1024
    return 4 * taps * (bn // 2) * 128 + 8 * 4096 + (2 * 4 + 9) * 8 + 16 + 1024 + 2 * halo


def _halo_fits(wl, bn):
    """Whether a forced tile width fits one CTA's shared memory (the host refuses the plan
    otherwise): stages of three taps for 64- and 128-wide tiles where they fit, else two."""
    return _halo_smem(wl, bn, 2) <= SMEM_LIMIT


@pytest.mark.parametrize("bn", [64, 128, 256])
@pytest.mark.parametrize("name", sorted(GEOMETRIES))
def test_halo_geometries_each_width(sg, name, bn):
    n, h, w_, c, k, r, s, pad, dil = GEOMETRIES[name]
    wl, x, w, b = _case(n, h, w_, c, k, r, s, pad, dil, seed=sum(map(ord, name)) % 1000)
    algo = make_algo(sg, loader=HALO, block_n=bn, wait_limit_ns=WAIT)
    if not _halo_fits(wl, bn):
        with pytest.raises(sg.Conv2dError) as e:
            gpu_conv(sg, x, w, b, wl.options(), algo=algo)
        assert e.value.code == 2  # CONV2D_ERR_UNSUPPORTED
        return
    _check(sg, wl, x, w, b, algo, f"{name} bn={bn}")


@pytest.mark.parametrize("split", [0, 3])
@pytest.mark.parametrize("name", sorted(GEOMETRIES))
def test_halo_tma_store_path(sg, name, split):
    """The TMA store path (a measurement hook), whole and cut tiles."""
    n, h, w_, c, k, r, s, pad, dil = GEOMETRIES[name]
    wl, x, w, b = _case(n, h, w_, c, k, r, s, pad, dil, seed=sum(map(ord, name)) % 991)
    algo = make_algo(sg, loader=HALO, wait_limit_ns=WAIT, debug_flags=sg.DEBUG_TMA_STORE, splits=split)
    try:
        _check(sg, wl, x, w, b, algo, f"{name} splits={split} TMA stores")
    except sg.Conv2dError as e:  # more splits than stages, or the halos do not fit
        assert e.code == 2


@pytest.mark.parametrize("name", ["n3_14x14_c128_k136", "n4_9x9_1x1_c192_k320", "n2_8x12_3x2_pad10_k48",
                                  "n1_16x16_5x5_c256_k128"])
def test_halo_integer_inputs_exact(sg, name):
    """Small integers: every product and partial sum is exact in fp32, so the result must equal
    the oracle's bit for bit."""
    n, h, w_, c, k, r, s, pad, dil = GEOMETRIES[name]
    wl, x, w, b = _case(n, h, w_, c, k, r, s, pad, dil, seed=3, dist="int:-3:3")
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=HALO, wait_limit_ns=WAIT))
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    assert np.array_equal(got.astype(np.float64), ref)


@pytest.fixture(scope="module")
def long_k():
    # 3 images of 14x14 (odd count), C = 256 (4 chunks x 5 two-tap stages = 20 stages per tile), K = 192.
    wl, x, w, b = _case(3, 14, 14, 256, 192, 3, 3, 1, 1, seed=11, dist="uniform")
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    return wl, x, w, b, ref


@pytest.mark.parametrize("reduction", [1, 2])
@pytest.mark.parametrize("split", [("splits", 2), ("splits", 7), ("splits", 16), ("grid", 3), ("grid", 5), ("grid", 23)])
def test_halo_cut_tiles_both_reductions(sg, long_k, split, reduction):
    wl, x, w, b, ref = long_k
    dev = torch.device("cuda", 0)
    params = sg.make_params(x.shape, w.shape, **wl.options())
    ws = torch.zeros(sg.workspace_bytes(params), dtype=torch.uint8, device=dev)
    algo = make_algo(sg, loader=HALO, wait_limit_ns=WAIT, reduction=reduction, **{split[0]: split[1]})
    got = gpu_conv(sg, x, w, b, wl.options(), algo=algo, workspace=ws)
    check_close(got, ref, wl.c, wl.r, wl.s, f"halo {split} reduction {reduction}")
    assert int(torch.count_nonzero(ws)) == 0
    assert sg.status(ws) == 0


def test_halo_ordered_reduction_reproducible(sg, long_k):
    wl, x, w, b, _ = long_k
    algo = make_algo(sg, loader=HALO, grid=5, reduction=1, wait_limit_ns=WAIT)
    first = gpu_conv(sg, x, w, b, wl.options(), algo=algo)
    again = gpu_conv(sg, x, w, b, wl.options(), algo=algo)
    assert np.array_equal(first, again)


@pytest.mark.parametrize("reduction", [1, 2])
def test_halo_bounded_wait_reports_timeout_and_recovers(sg, long_k, reduction):
    wl, x, w, b, ref = long_k
    dev = torch.device("cuda", 0)
    params = sg.make_params(x.shape, w.shape, **wl.options())
    ws = torch.zeros(sg.workspace_bytes(params), dtype=torch.uint8, device=dev)
    hook = make_algo(sg, loader=HALO, splits=3, debug_flags=sg.DEBUG_SKIP_SIGNAL, wait_limit_ns=20_000_000,
                     reduction=reduction)
    gpu_conv(sg, x, w, b, wl.options(), algo=hook, workspace=ws)
    assert sg.status(ws) == 6  # CONV2D_ERR_TIMEOUT
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=HALO, splits=3, wait_limit_ns=WAIT),
                   workspace=ws)
    check_close(got, ref, wl.c, wl.r, wl.s, "after timeout")
    assert sg.status(ws) == 0


@pytest.mark.parametrize("mode", [(True, False), (False, True), (True, True)])
@pytest.mark.parametrize("name", ["n3_14x14_c128_k136", "n2_10x10_c64_k80"])
def test_halo_fused_epilogue_whole_tiles(sg, name, mode):
    n, h, w_, c, k, r, s, pad, dil = GEOMETRIES[name]
    wl, x, w, b = _case(n, h, w_, c, k, r, s, pad, dil, seed=5)
    got = gpu_conv_epi(sg, x, w, b, wl.options(), *mode, algo=make_algo(sg, loader=HALO, wait_limit_ns=WAIT))
    u = oracle.conv2d_fwd(x, w, b, **wl.options())
    check_epilogue(got.astype(np.float64), u, wl.c, wl.r, wl.s, *mode, f"{name} fused {mode}")


# Groups on the halo kernel (n, h, w, c, k, r, s, pad, dil, groups): one and two chunks per
# group, an odd image count, a group narrower than the tile (its block reads the next group's
# weight rows and stores only its own columns), a group width that is not a tile multiple,
# dilation and 1x1.
GROUPED = {
    "g2_cg64_kg64": (2, 10, 10, 128, 128, 3, 3, 1, 1, 2),
    "g4_cg64_kg128_n3": (3, 13, 11, 256, 512, 3, 3, 1, 1, 4),
    "g2_cg128_kg96_dil2": (1, 9, 12, 256, 192, 3, 3, 2, 2, 2),
    "g8_cg64_kg64_1x1": (3, 8, 8, 512, 512, 1, 1, 0, 1, 8),
    "g4_cg64_kg16": (2, 7, 7, 256, 64, 3, 3, 1, 1, 4),
}


@pytest.mark.parametrize("split", [0, 3])
@pytest.mark.parametrize("name", sorted(GROUPED))
def test_halo_grouped(sg, name, split):
    """Column blocks never straddle a group; each group's halos start at its first input
    channel and its weight boxes at its own rows; whole and cut tiles."""
    n, h, w_, c, k, r, s, pad, dil, groups = GROUPED[name]
    wl, x, w, b = _case(n, h, w_, c, k, r, s, pad, dil, seed=sum(map(ord, name)) % 997, groups=groups)
    algo = make_algo(sg, loader=HALO, wait_limit_ns=WAIT, splits=split)
    stages = (c // groups // 64) * -(-(r * s) // 3)  # at most this many (three taps per stage)
    if split > stages:
        with pytest.raises(sg.Conv2dError) as e:
            gpu_conv(sg, x, w, b, wl.options(), algo=algo)
        assert e.value.code == 2
        return
    _check(sg, wl, x, w, b, algo, f"halo grouped {name} splits={split}")


def test_halo_grouped_integer_exact(sg):
    wl, x, w, b = _case(3, 9, 10, 256, 256, 3, 3, 1, 1, seed=7, dist="int:-3:3", groups=4)
    got = gpu_conv(sg, x, w, b, wl.options(), algo=make_algo(sg, loader=HALO, wait_limit_ns=WAIT))
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    assert np.array_equal(got.astype(np.float64), ref)


@pytest.mark.parametrize("shape", [
    (1, 8, 8, 64, 64, 3, 3, 2, 1, 1, 1),    # stride 2
    (1, 8, 8, 32, 64, 3, 3, 1, 1, 1, 1),    # C % 64 != 0
    (1, 8, 300, 64, 64, 3, 3, 1, 1, 1, 1),  # padded row longer than a TMA box dimension
    (1, 8, 8, 128, 64, 3, 3, 1, 1, 1, 4),   # groups of 32 channels
])
def test_halo_refuses_ineligible_shapes(sg, shape):
    n, h, w_, c, k, r, s, stride, pad, dil, groups = shape
    dev = torch.device("cuda", 0)
    x = torch.zeros((n, h, w_, c), dtype=torch.bfloat16, device=dev)
    w = torch.zeros((k, r, s, c // groups), dtype=torch.bfloat16, device=dev)
    with pytest.raises(sg.Conv2dError) as e:
        sg.conv2d_fwd(x, w, None, stride, pad, dil, groups, algo=make_algo(sg, loader=HALO))
    assert e.value.code == 2


@pytest.mark.parametrize("name", ["resnet_56x56_c64", "resnet_28x28_c256", "splitk_7x7_c2048", "dil2_64_c128",
                                  "grouped_28x28_c512_g8"])
def test_halo_full_size_workloads(sg, name):
    wl = workloads.get(name)
    x, w, b = workloads.make_inputs(wl)
    _check(sg, wl, x, w, b, make_algo(sg, loader=HALO, wait_limit_ns=WAIT), name + " halo")
    assert sg.last_launch_count() == 1
