"""The TMA-descriptor cache of the forward calls: a repeated call with the same pointers
and shape reuses its tensor maps, and a changed pointer or shape encodes new ones; every
call stays at parity with the oracle (a stale map would read the old buffer or the old
geometry).  Needs a GB300."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import split_gemm_gb300
    split_gemm_gb300.load_library()
    torch.cuda.set_device(0)
    return split_gemm_gb300


def _case(n, h, w, seed):
    wl = workloads.Workload(f"cache{seed}", n, h, w, 64, 64, 3, 3, 1, 1, 1, 1, 1, 1, x_dist="normal", w_dist="he",
                            bias="normal:0.1", seed=seed)
    x, wt, b = workloads.make_inputs(wl)
    return wl, x, wt, b


def _run(sg, wl, xd, wd, bd):
    y = sg.conv2d_fwd(xd, wd, bd, **wl.options())
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _check(wl, got, x, w, b, what):
    check_close(got, oracle.conv2d_fwd(x, w, b, **wl.options()), wl.c, wl.r, wl.s, what)


def test_map_cache_hits_and_reencodes(sg):
    dev = torch.device("cuda", 0)
    wl, x, w, b = _case(2, 14, 14, 31)
    params = sg.make_params(x.shape, w.shape, **wl.options())
    assert sg.query_algo(params).loader in (sg.LOADER_TMA_IM2COL, sg.LOADER_TMA_PAIR)  # loaders that encode maps
    xd, wd, bd = x.to(dev), w.to(dev), b.to(dev)

    h0, m0 = sg.tensor_map_cache_stats()
    _check(wl, _run(sg, wl, xd, wd, bd), x, w, b, "first call")
    h1, m1 = sg.tensor_map_cache_stats()
    assert (h1, m1) == (h0, m0 + 1)  # fresh pointers: encoded

    _check(wl, _run(sg, wl, xd, wd, bd), x, w, b, "same pointers")
    h2, m2 = sg.tensor_map_cache_stats()
    assert (h2, m2) == (h1 + 1, m1)  # same pointers and shape: reused

    # Same pointers, new contents: the cached maps still read the buffers as they are now.
    _, x_new, w_new, _ = _case(2, 14, 14, 32)
    xd.copy_(x_new.to(dev))
    wd.copy_(w_new.to(dev))
    _check(wl, _run(sg, wl, xd, wd, bd), x_new, w_new, b, "same pointers, new contents")
    h3, m3 = sg.tensor_map_cache_stats()
    assert (h3, m3) == (h2 + 1, m2)

    # A new activation buffer (other data): new maps, and the result follows the new buffer.
    xd2 = x.to(dev)
    assert xd2.data_ptr() != xd.data_ptr()
    _check(wl, _run(sg, wl, xd2, wd, bd), x, w_new, b, "new x pointer")
    h4, m4 = sg.tensor_map_cache_stats()
    assert (h4, m4) == (h3, m3 + 1)

    # A new weight buffer.
    wd2 = w.to(dev)
    _check(wl, _run(sg, wl, xd2, wd2, bd), x, w, b, "new w pointer")
    h5, m5 = sg.tensor_map_cache_stats()
    assert (h5, m5) == (h4, m4 + 1)


def test_map_cache_shape_change_at_same_address(sg):
    """A different shape on the same allocation (a view of fewer images, then a different
    spatial size carved from the same storage) is a different key and encodes afresh."""
    dev = torch.device("cuda", 0)
    wl, x, w, b = _case(4, 12, 12, 41)
    xd, wd, bd = x.to(dev), w.to(dev), b.to(dev)
    _check(wl, _run(sg, wl, xd, wd, bd), x, w, b, "n=4")
    h0, m0 = sg.tensor_map_cache_stats()

    wl2 = workloads.Workload("cache_n2", 2, 12, 12, 64, 64, 3, 3, 1, 1, 1, 1, 1, 1, x_dist="normal", w_dist="he",
                             bias="normal:0.1", seed=41)
    got = _run(sg, wl2, xd[:2], wd, bd)  # same base address, two images
    _check(wl2, got, x[:2], w, b, "n=2 view")
    h1, m1 = sg.tensor_map_cache_stats()
    assert (h1, m1) == (h0, m0 + 1)

    flat = xd.reshape(-1)[: 3 * 10 * 10 * 64].view(3, 10, 10, 64)  # same address, other geometry
    wl3 = workloads.Workload("cache_10", 3, 10, 10, 64, 64, 3, 3, 1, 1, 1, 1, 1, 1, x_dist="normal", w_dist="he",
                             bias="normal:0.1", seed=41)
    got = _run(sg, wl3, flat, wd, bd)
    _check(wl3, got, flat.cpu(), w, b, "10x10 view")
    h2, m2 = sg.tensor_map_cache_stats()
    assert (h2, m2) == (h1, m1 + 1)
    assert np.isfinite(got).all()
