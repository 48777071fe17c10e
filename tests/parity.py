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


def check_epilogue(got, u, c, r, s, relu_on, out_bf16, what=""):
    """Fused-epilogue parity: ``got`` (the kernel's output, widened to float64) must lie in
    the range the epilogue maps [u - B, u + B] to, where u is the oracle's exact value
    before the epilogue and B the fp32 parity bound 1e-5*|u| + 1e-4*sqrt(C*R*S).

    ReLU and the bf16 rounding are monotone, so the kernel's fp32 value f, |f - u| <= B,
    can only produce an output inside that range; with a bf16 output the range is a
    single value wherever [u - B, u + B] rounds one way, and the output must equal it.
    Returns the fraction of elements whose output the range determines exactly.
    """
    from oracle import epilogue
    got = np.asarray(got, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    assert got.shape == u.shape, f"{what}: shape {got.shape} vs {u.shape}"
    if got.size == 0:
        return 1.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rtol, atol = oracle.tolerance(c, r, s)
    lo, hi = epilogue.bracket(u, rtol * np.abs(u) + atol, relu_on, out_bf16)
    bad = (got < lo) | (got > hi)
    if np.any(bad):
        i = int(np.flatnonzero(bad.reshape(-1))[0])
        raise AssertionError(
            f"{what}: element {np.unravel_index(i, got.shape)} got {got.flat[i]!r} outside "
            f"[{lo.flat[i]!r}, {hi.flat[i]!r}] (u {u.flat[i]!r}); {int(np.count_nonzero(bad))} of {got.size} bad")
    return float(np.count_nonzero(lo == hi)) / got.size


def gpu_conv_epi(sg, x, w, b, opts, relu_on, out_bf16, algo=None, fill=float("nan"), workspace=None):
    """The fused call through the binding; y is pre-filled so that unwritten elements show."""
    dev = torch.device("cuda", 0)
    params = sg.make_params(x.shape, w.shape, **opts)
    p, q = sg.output_shape(params)
    y = torch.full((params.n, p, q, params.k), fill, dtype=torch.bfloat16 if out_bf16 else torch.float32,
                   device=dev)
    sg.conv2d_fwd_into(y, x.to(dev), w.to(dev), None if b is None else b.to(dev), **opts, algo=algo,
                       relu=relu_on, workspace=workspace)
    torch.cuda.synchronize()
    return y.cpu().to(torch.float64).numpy()
