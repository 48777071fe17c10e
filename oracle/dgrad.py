"""CPU fp64 reference for the data (input) gradient of 2-D convolution -- TEST INFRASTRUCTURE ONLY.

Only ``tests/`` and the CPU-baseline leg of ``bench.py`` may use this module.  It
shares no code with the CUDA path in ``split_gemm_gb300``.

The arithmetic is ``conv2d_dgrad.c`` (plain C, POSIX threads): the derivative of
the forward sum with respect to the input, which burn computes as
``conv_data_backward`` (docs.rs burn-cubecl 0.20.0,
``burn_cubecl/kernel/conv/base.rs``; output gradient NHWC, weights KRSC, input
gradient NHWC) -- also conv_transpose2d's definition::

    dx[n][h][w][ci] = sum_{r,s,k} dy[n][p][q][k] * w[k][r][s][ci - g*C/G]
        where h + ph - r*dh = p*sh and w + pw - s*dw = q*sw (0 <= p < P, 0 <= q < Q)

Pinned by ``tests/test_oracle_dgrad.py``: the adjoint identity against the
(separately pinned) forward oracle, a library gradient, 1x1 = matmul, a col2im
brute force with integer inputs, and planted mutants.
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
_SRC = os.path.join(_HERE, "conv2d_dgrad.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle_dgrad.so")
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
    lib.oracle_dgrad_f64.restype = ctypes.c_int
    lib.oracle_dgrad_f64.argtypes = [i64p, i64p, vp, vp, vp, vp, ctypes.c_int]
    lib.oracle_dgrad_bf16.restype = ctypes.c_int
    lib.oracle_dgrad_bf16.argtypes = [i64p, i64p, vp, vp, vp, vp, ctypes.c_int]
    lib.oracle_dgrad_points_f64.restype = ctypes.c_int
    lib.oracle_dgrad_points_f64.argtypes = [i64p, i64p, vp, vp, vp, vp, ctypes.c_int64, vp, vp]
    return lib


def load(path: Optional[str] = None):
    global _lib
    if path is not None:
        return _bind(path)
    with _lock:
        if _lib is None:
            _lib = _bind(build())
        return _lib


def _shapes(x_shape, dyshape, wshape, stride, padding, dilation, groups):
    """(dims, opts) from the input shape [N,H,W,C], dy [N,P,Q,K] and the weight shape [K,R,S,C/G]."""
    (n, h, w, c, k, r, s), (sh, sw, ph, pw, dh, dw), dims, opts = _dims_opts(x_shape, wshape, stride, padding,
                                                                            dilation, groups)
    p, q = out_extent(h, ph, dh, r, sh), out_extent(w, pw, dw, s, sw)
    if tuple(dyshape) != (n, p, q, k):
        raise ValueError(f"dy must be [{n}, {p}, {q}, {k}], got {list(dyshape)}")
    return dims, opts


def conv2d_dgrad(dy, w, x_shape, stride=1, padding=0, dilation=1, groups=1, *, threads: Optional[int] = None,
                 with_mass: bool = False, lib=None):
    """Input gradient over bf16 dy [N,P,Q,K] and w [K,R,S,C/groups] (torch tensors or uint16 bit arrays)
    for a forward convolution of an input of shape ``x_shape`` [N,H,W,C].

    Returns dx [N,H,W,C] float64, and with ``with_mass`` also the per-element sum of |terms|."""
    lib = lib or load()
    dys, ws = _bf16_bits(dy), _bf16_bits(w)
    dims, opts = _shapes(x_shape, dys.shape, ws.shape, stride, padding, dilation, groups)
    dx = np.zeros(tuple(int(v) for v in x_shape), dtype=np.float64)
    mass = np.zeros_like(dx) if with_mass else None
    rc = lib.oracle_dgrad_bf16(dims, opts, _ptr(dys), _ptr(ws), _ptr(dx), _ptr(mass), threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_dgrad_bf16 failed with code {rc}")
    return (dx, mass) if with_mass else dx


def conv2d_dgrad_f64(dy: np.ndarray, w: np.ndarray, x_shape, stride=1, padding=0, dilation=1, groups=1, *,
                     threads: Optional[int] = None, lib=None) -> np.ndarray:
    """As conv2d_dgrad over float64 inputs (no bf16 widening), for exact pins."""
    lib = lib or load()
    dys = np.ascontiguousarray(dy, dtype=np.float64)
    ws = np.ascontiguousarray(w, dtype=np.float64)
    dims, opts = _shapes(x_shape, dys.shape, ws.shape, stride, padding, dilation, groups)
    dx = np.zeros(tuple(int(v) for v in x_shape), dtype=np.float64)
    rc = lib.oracle_dgrad_f64(dims, opts, _ptr(dys), _ptr(ws), _ptr(dx), None, threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_dgrad_f64 failed with code {rc}")
    return dx


def conv2d_dgrad_points_f64(dy: np.ndarray, w: np.ndarray, x_shape, stride, padding, dilation,
                            m_idx: Sequence[int], c_idx: Sequence[int], groups=1,
                            lib=None) -> Tuple[np.ndarray, np.ndarray]:
    """Selected elements dx[m][c] of the gradient viewed as [N*H*W][C] and their |term| sums,
    over float64 inputs."""
    lib = lib or load()
    dys = np.ascontiguousarray(dy, dtype=np.float64)
    ws = np.ascontiguousarray(w, dtype=np.float64)
    dims, opts = _shapes(x_shape, dys.shape, ws.shape, stride, padding, dilation, groups)
    mi = np.ascontiguousarray(m_idx, dtype=np.int64)
    ci = np.ascontiguousarray(c_idx, dtype=np.int64)
    if mi.shape != ci.shape:
        raise ValueError("m_idx and c_idx must have the same length")
    out = np.zeros(mi.shape, dtype=np.float64)
    mass = np.zeros(mi.shape, dtype=np.float64)
    rc = lib.oracle_dgrad_points_f64(dims, opts, _ptr(dys), _ptr(ws), _ptr(mi), _ptr(ci), int(mi.size), _ptr(out),
                                     _ptr(mass))
    if rc != 0:
        raise ValueError(f"oracle_dgrad_points_f64 failed with code {rc}")
    return out, mass
