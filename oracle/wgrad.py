"""CPU fp64 reference for the weight gradient of 2-D convolution -- TEST INFRASTRUCTURE ONLY.

Only ``tests/`` and the CPU-baseline leg of ``bench.py`` may use this module.  It
shares no code with the CUDA path in ``split_gemm_gb300``.

The arithmetic is ``conv2d_wgrad.c`` (plain C, POSIX threads): the derivative of
the forward sum with respect to the weight, which burn computes as
``conv_weight_backward`` (docs.rs burn-cubecl 0.20.0,
``burn_cubecl/kernel/conv/base.rs``; input and output gradient NHWC, weight
gradient [K][R][S][C/groups])::

    dw[k][r][s][c] = sum_{n,p,q} dy[n][p][q][k] * x[n][p*sh-ph+r*dh][q*sw-pw+s*dw][g*C/G + c]

Pinned by ``tests/test_oracle_wgrad.py``: the adjoint identity against the
(separately pinned) forward oracle, a library gradient, 1x1 = matmul, an
explicit im2col brute force with integer inputs, and planted mutants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence, Tuple

import numpy as np

from . import _bf16_bits, _dims_opts, _ptr, default_threads, out_extent

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv2d_wgrad.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle_wgrad.so")
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math"]

_lock = threading.Lock()
_lib = None


def compile_library(src: str = _SRC, out: str = _LIB_PATH) -> str:
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *_CFLAGS, src, "-o", tmp], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_library()
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    i64p = ctypes.POINTER(ctypes.c_int64)
    vp = ctypes.c_void_p
    lib.oracle_wgrad_f64.restype = ctypes.c_int
    lib.oracle_wgrad_f64.argtypes = [i64p, i64p, vp, vp, vp, vp, ctypes.c_int]
    lib.oracle_wgrad_bf16.restype = ctypes.c_int
    lib.oracle_wgrad_bf16.argtypes = [i64p, i64p, vp, vp, vp, vp, ctypes.c_int]
    lib.oracle_wgrad_points_f64.restype = ctypes.c_int
    lib.oracle_wgrad_points_f64.argtypes = [i64p, i64p, vp, vp, vp, vp, ctypes.c_int64, vp, vp]
    return lib


def load(path: Optional[str] = None):
    global _lib
    if path is not None:
        return _bind(path)
    with _lock:
        if _lib is None:
            _lib = _bind(build())
        return _lib


def _shapes(xshape, dyshape, wshape, stride, padding, dilation, groups):
    """(dims, opts, w-gradient shape) from x [N,H,W,C], dy [N,P,Q,K] and the weight shape [K,R,S,C/G]."""
    (n, h, w, c, k, r, s), (sh, sw, ph, pw, dh, dw), dims, opts = _dims_opts(xshape, wshape, stride, padding,
                                                                            dilation, groups)
    p, q = out_extent(h, ph, dh, r, sh), out_extent(w, pw, dw, s, sw)
    if tuple(dyshape) != (n, p, q, k):
        raise ValueError(f"dy must be [{n}, {p}, {q}, {k}], got {list(dyshape)}")
    return dims, opts, (k, r, s, c // groups)


def conv2d_wgrad(x, dy, w_shape, stride=1, padding=0, dilation=1, groups=1, *, threads: Optional[int] = None,
                 with_mass: bool = False, lib=None):
    """Weight gradient over bf16 x [N,H,W,C] and dy [N,P,Q,K] (torch tensors or uint16 bit arrays).

    Returns dw [K,R,S,C/groups] float64, and with ``with_mass`` also the per-element
    sum of |terms| of the same shape."""
    lib = lib or load()
    xs, dys = _bf16_bits(x), _bf16_bits(dy)
    dims, opts, shape = _shapes(xs.shape, dys.shape, w_shape, stride, padding, dilation, groups)
    dw = np.zeros(shape, dtype=np.float64)
    mass = np.zeros(shape, dtype=np.float64) if with_mass else None
    rc = lib.oracle_wgrad_bf16(dims, opts, _ptr(xs), _ptr(dys), _ptr(dw), _ptr(mass), threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_wgrad_bf16 failed with code {rc}")
    return (dw, mass) if with_mass else dw


def conv2d_wgrad_f64(x: np.ndarray, dy: np.ndarray, w_shape, stride=1, padding=0, dilation=1, groups=1, *,
                     threads: Optional[int] = None, lib=None) -> np.ndarray:
    """As conv2d_wgrad over float64 inputs (no bf16 widening), for exact pins."""
    lib = lib or load()
    xs = np.ascontiguousarray(x, dtype=np.float64)
    dys = np.ascontiguousarray(dy, dtype=np.float64)
    dims, opts, shape = _shapes(xs.shape, dys.shape, w_shape, stride, padding, dilation, groups)
    dw = np.zeros(shape, dtype=np.float64)
    rc = lib.oracle_wgrad_f64(dims, opts, _ptr(xs), _ptr(dys), _ptr(dw), None, threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_wgrad_f64 failed with code {rc}")
    return dw


def conv2d_wgrad_points_f64(x: np.ndarray, dy: np.ndarray, w_shape, stride, padding, dilation,
                            k_idx: Sequence[int], j_idx: Sequence[int], groups=1,
                            lib=None) -> Tuple[np.ndarray, np.ndarray]:
    """Selected elements dw[k][j] of the gradient viewed as [K][R*S*C/groups] and their |term| sums,
    over float64 inputs (widen once with ``oracle.widen_bf16``, sample many times)."""
    lib = lib or load()
    xs = np.ascontiguousarray(x, dtype=np.float64)
    dys = np.ascontiguousarray(dy, dtype=np.float64)
    dims, opts, _ = _shapes(xs.shape, dys.shape, w_shape, stride, padding, dilation, groups)
    ki = np.ascontiguousarray(k_idx, dtype=np.int64)
    ji = np.ascontiguousarray(j_idx, dtype=np.int64)
    if ki.shape != ji.shape:
        raise ValueError("k_idx and j_idx must have the same length")
    out = np.zeros(ki.shape, dtype=np.float64)
    mass = np.zeros(ki.shape, dtype=np.float64)
    rc = lib.oracle_wgrad_points_f64(dims, opts, _ptr(xs), _ptr(dys), _ptr(ki), _ptr(ji), int(ki.size), _ptr(out),
                                     _ptr(mass))
    if rc != 0:
        raise ValueError(f"oracle_wgrad_points_f64 failed with code {rc}")
    return out, mass
