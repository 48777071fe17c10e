"""Random layers large enough for the heuristic to pick the CTA-pair kernels (the im2col pair
kernel with its own schedule, groups of 64+ channels, block-diagonal tiles) or to keep the
one-CTA kernel, checked element by element against the CPU oracle through the C ABI with no
plan forced (needs a GB300).  Shapes are drawn from a seeded generator."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import check_close, gpu_conv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import split_gemm_gb300
    split_gemm_gb300.load_library()
    torch.cuda.set_device(0)
    return split_gemm_gb300


def _draw(seed):
    g = torch.Generator("cpu")
    g.manual_seed(20_000 + seed)

    def pick(seq):
        return seq[int(torch.randint(0, len(seq), (1,), generator=g))]

    while True:
        groups = pick([1, 1, 1, 2, 4, 32])
        cg = 8 if groups == 32 else pick([64, 128, 128])
        c = cg * groups
        kg = 8 if groups == 32 else pick([64, 96, 128, 256])
        k = kg * groups
        n = pick([4, 8, 8, 16])
        h = pick([14, 17, 22, 28, 31])
        w = pick([14, 19, 28, 30])
        r = pick([1, 3, 3, 5])
        s = r if pick([0, 1]) else pick([1, 3])
        st = pick([1, 1, 1, 2])
        dil = pick([1, 1, 2]) if st == 1 else 1
        ph, pw = (dil * (r - 1)) // 2, (dil * (s - 1)) // 2
        if h + 2 * ph >= dil * (r - 1) + 1 and w + 2 * pw >= dil * (s - 1) + 1:
            break
    return workloads.Workload(f"auto{seed}", n, h, w, c, k, r, s, st, st, ph, pw, dil, dil, x_dist="normal",
                              w_dist="he", bias="normal:0.1" if seed % 2 == 0 else None, seed=seed, groups=groups)


@pytest.mark.parametrize("seed", range(16))
def test_auto_plans_random_layers(sg, seed):
    wl = _draw(seed)
    x, w, b = workloads.make_inputs(wl)
    params = sg.make_params(x.shape, w.shape, **wl.options())
    plan = sg.query_algo(params)
    got = gpu_conv(sg, x, w, b, wl.options())
    ref = oracle.conv2d_fwd(x, w, b, **wl.options())
    check_close(got, ref, wl.c // wl.groups, wl.r, wl.s, f"{wl.describe()} plan {plan.loader}")


def test_auto_plans_cover_the_pair_kernels(sg):
    """The draw above reaches a CTA-pair kernel and the block-diagonal tiles (so a change of
    the rules that stopped exercising them would show here rather than pass silently; the
    workload tests run both pair kernels at full size: the im2col one on the 56x56, split-K,
    projection and grouped layers, the halo one on the 28x28 and dilated layers, and forced on
    the grouped layer)."""
    loaders = set()
    for seed in range(16):
        wl = _draw(seed)
        loaders.add(sg.query_algo(sg.make_params((wl.n, wl.h, wl.w, wl.c), (wl.k, wl.r, wl.s, wl.c // wl.groups),
                                                 **wl.options())).loader)
    assert sg.LOADER_BLOCKDIAG in loaders and loaders & {sg.LOADER_TMA_PAIR, sg.LOADER_PAIR_HALO}, loaders
