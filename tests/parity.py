"""Parity helpers: run the CUDA path through the C ABI and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle


def check_close(got, ref, c, r, s, what=""):
    """Element-wise |got - ref| <= 1e-5*|ref| + 1e-4*sqrt(C*R*S); raises with the worst element."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    if got.size == 0:
        return 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rtol, atol = oracle.tolerance(c, r, s)
    err = np.abs(got - ref)
    bound = rtol * np.abs(ref) + atol
    ratio = err / bound
    worst = int(np.argmax(ratio))
    assert ratio.flat[worst] <= 1.0, (
        f"{what}: element {np.unravel_index(worst, got.shape)} got {got.flat[worst]!r} ref {ref.flat[worst]!r} "
        f"err {err.flat[worst]:.3e} > bound {bound.flat[worst]:.3e}; "
        f"{int(np.count_nonzero(ratio > 1))} of {got.size} elements out of tolerance")
    return float(ratio.max())


def gpu_conv(sg, x, w, b, opts, algo=None, workspace=None):
    dev = torch.device("cuda", 0)
    y = sg.conv2d_fwd(x.to(dev), w.to(dev), None if b is None else b.to(dev), **opts, algo=algo,
                      workspace=workspace)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def make_algo(sg, block_n=0, splits=0, loader=0, debug_flags=0, wait_limit_ns=0, block_m=0, grid=0, reduction=0):
    a = sg.Algo()
    a.block_n, a.splits, a.loader, a.block_m, a.grid = block_n, splits, loader, block_m, grid
    a.debug_flags, a.wait_limit_ns, a.reduction = debug_flags, wait_limit_ns, reduction
    return a
