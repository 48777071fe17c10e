"""CPU fp64 reference for 2-D convolution forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA path in
``split_gemm_gb300`` and never imports it.

The arithmetic lives in ``conv2d_direct.c`` (plain C, POSIX threads): the
seven-loop direct convolution that burn keeps as its ``Direct`` strategy
(docs.rs burn-cubecl 0.20.0, ``burn_cubecl/kernel/conv/base.rs``,
``ConvStrategy``), which the im2col and implicit-GEMM algorithms of burn PR
#2287 ("Changes") and burn PR #2545 ("Changes") compute by other means.  This
module only builds that library with ``gcc`` and marshals arguments.

Pinned by ``tests/test_oracle_pins.py`` (delta kernels, 1x1 = matmul,
explicit im2col + GEMM brute force with exact integer arithmetic, a library
convolution, linearity/bias invariants, a hand-worked fixture) and
``tests/test_oracle_mutations.py`` (each planted mistake fails a pin).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv2d_direct.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_conv2d.so")
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math"]

_lock = threading.Lock()
_lib = None


def compile_library(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``src`` into the shared library ``out`` with gcc and return its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *_CFLAGS, src, "-o", tmp], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_library()
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    i64p = ctypes.POINTER(ctypes.c_int64)
    vp = ctypes.c_void_p
    lib.oracle_out_extent.restype = ctypes.c_int64
    lib.oracle_out_extent.argtypes = [ctypes.c_int64] * 5
    lib.oracle_conv2d_f64.restype = ctypes.c_int
    lib.oracle_conv2d_f64.argtypes = [i64p, i64p, vp, vp, vp, vp, ctypes.c_int]
    lib.oracle_conv2d_bf16.restype = ctypes.c_int
    lib.oracle_conv2d_bf16.argtypes = [i64p, i64p, vp, vp, vp, vp, ctypes.c_int]
    lib.oracle_conv2d_points_bf16.restype = ctypes.c_int
    lib.oracle_conv2d_points_bf16.argtypes = [i64p, i64p, vp, vp, vp, vp, vp, ctypes.c_int64, vp]
    lib.oracle_conv2d_points_f64.restype = ctypes.c_int
    lib.oracle_conv2d_points_f64.argtypes = [i64p, i64p, vp, vp, vp, vp, vp, ctypes.c_int64, vp]
    return lib


def load(path: Optional[str] = None):
    """Return the bound library (building the default one on first use)."""
    global _lib
    if path is not None:
        return _bind(path)
    with _lock:
        if _lib is None:
            _lib = _bind(build())
        return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _pair(v) -> Tuple[int, int]:
    if isinstance(v, (tuple, list)):
        return int(v[0]), int(v[1])
    return int(v), int(v)


def out_extent(in_size: int, pad: int, dil: int, ker: int, stride: int, lib=None) -> int:
    """Output size along one axis: floor((in + 2*pad - dil*(ker-1) - 1)/stride) + 1, or 0."""
    lib = lib or load()
    return int(lib.oracle_out_extent(in_size, pad, dil, ker, stride))


def _bf16_bits(t) -> np.ndarray:
    """bf16 tensor/array -> contiguous uint16 numpy array of its bit patterns."""
    if isinstance(t, np.ndarray):
        if t.dtype != np.uint16:
            raise TypeError("numpy input must hold bf16 bit patterns as uint16")
        return np.ascontiguousarray(t)
    import torch
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bfloat16 tensor")
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _bias_f32(b) -> Optional[np.ndarray]:
    if b is None:
        return None
    if isinstance(b, np.ndarray):
        return np.ascontiguousarray(b, dtype=np.float32)
    return np.ascontiguousarray(b.detach().cpu().to(dtype=__import__("torch").float32).numpy())


def _dims_opts(xshape, wshape, stride, padding, dilation, groups=1):
    n, h, w, c = (int(v) for v in xshape)
    k, r, s, cg = (int(v) for v in wshape)
    groups = int(groups)
    if groups < 1 or c % groups or k % groups:
        raise ValueError(f"groups={groups} must divide C={c} and K={k}")
    if cg * groups != c:
        raise ValueError(f"channel mismatch: input C={c}, weight C/groups={cg}, groups={groups}")
    sh, sw = _pair(stride)
    ph, pw = _pair(padding)
    dh, dw = _pair(dilation)
    dims = (ctypes.c_int64 * 7)(n, h, w, c, k, r, s)
    opts = (ctypes.c_int64 * 7)(sh, sw, ph, pw, dh, dw, groups)
    return (n, h, w, c, k, r, s), (sh, sw, ph, pw, dh, dw), dims, opts


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def conv2d_fwd(x, w, bias=None, stride=1, padding=0, dilation=1, threads: Optional[int] = None,
               lib=None, groups=1) -> np.ndarray:
    """Direct convolution over bf16 inputs in fp64.

    x: [N,H,W,C] bf16 (torch tensor or uint16 bit array); w: [K,R,S,C/groups] bf16;
    bias: [K] fp32 or None.  Returns y: [N,P,Q,K] float64 (NHWC).
    """
    lib = lib or load()
    xs = _bf16_bits(x)
    ws = _bf16_bits(w)
    b = _bias_f32(bias)
    (n, h, wd, c, k, r, s), (sh, sw, ph, pw, dh, dw), dims, opts = _dims_opts(xs.shape, ws.shape, stride,
                                                                              padding, dilation, groups)
    p = out_extent(h, ph, dh, r, sh, lib)
    q = out_extent(wd, pw, dw, s, sw, lib)
    y = np.zeros((n, p, q, k), dtype=np.float64)
    rc = lib.oracle_conv2d_bf16(dims, opts, _ptr(xs), _ptr(ws), _ptr(b), _ptr(y),
                                threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_conv2d_bf16 failed with code {rc}")
    return y


def conv2d_fwd_f64(x: np.ndarray, w: np.ndarray, bias=None, stride=1, padding=0, dilation=1,
                   threads: Optional[int] = None, lib=None, groups=1) -> np.ndarray:
    """Direct convolution over float64 inputs (no bf16 widening), for exact pins."""
    lib = lib or load()
    xs = np.ascontiguousarray(x, dtype=np.float64)
    ws = np.ascontiguousarray(w, dtype=np.float64)
    b = _bias_f32(bias)
    (n, h, wd, c, k, r, s), (sh, sw, ph, pw, dh, dw), dims, opts = _dims_opts(xs.shape, ws.shape, stride,
                                                                              padding, dilation, groups)
    p = out_extent(h, ph, dh, r, sh, lib)
    q = out_extent(wd, pw, dw, s, sw, lib)
    y = np.zeros((n, p, q, k), dtype=np.float64)
    rc = lib.oracle_conv2d_f64(dims, opts, _ptr(xs), _ptr(ws), _ptr(b), _ptr(y),
                               threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_conv2d_f64 failed with code {rc}")
    return y


def conv2d_fwd_points(x, w, bias, stride, padding, dilation, m_idx: Sequence[int],
                      k_idx: Sequence[int], lib=None, groups=1) -> np.ndarray:
    """Selected outputs y[m][k] of the [N*P*Q, K] view of the NHWC output, in float64."""
    lib = lib or load()
    xs = _bf16_bits(x)
    ws = _bf16_bits(w)
    b = _bias_f32(bias)
    _, _, dims, opts = _dims_opts(xs.shape, ws.shape, stride, padding, dilation, groups)
    mi = np.ascontiguousarray(m_idx, dtype=np.int64)
    ki = np.ascontiguousarray(k_idx, dtype=np.int64)
    if mi.shape != ki.shape:
        raise ValueError("m_idx and k_idx must have the same length")
    out = np.zeros(mi.shape, dtype=np.float64)
    rc = lib.oracle_conv2d_points_bf16(dims, opts, _ptr(xs), _ptr(ws), _ptr(b), _ptr(mi), _ptr(ki),
                                       int(mi.size), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_conv2d_points_bf16 failed with code {rc}")
    return out


def conv2d_fwd_points_f64(x: np.ndarray, w: np.ndarray, bias, stride, padding, dilation, m_idx, k_idx,
                          lib=None, groups=1) -> np.ndarray:
    """As conv2d_fwd_points over float64 inputs (widen once, sample many times)."""
    lib = lib or load()
    xs = np.ascontiguousarray(x, dtype=np.float64)
    ws = np.ascontiguousarray(w, dtype=np.float64)
    b = _bias_f32(bias)
    _, _, dims, opts = _dims_opts(xs.shape, ws.shape, stride, padding, dilation, groups)
    mi = np.ascontiguousarray(m_idx, dtype=np.int64)
    ki = np.ascontiguousarray(k_idx, dtype=np.int64)
    if mi.shape != ki.shape:
        raise ValueError("m_idx and k_idx must have the same length")
    out = np.zeros(mi.shape, dtype=np.float64)
    rc = lib.oracle_conv2d_points_f64(dims, opts, _ptr(xs), _ptr(ws), _ptr(b), _ptr(mi), _ptr(ki),
                                      int(mi.size), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_conv2d_points_f64 failed with code {rc}")
    return out


def widen_bf16(t) -> np.ndarray:
    """bf16 tensor -> float64 array holding exactly the same values."""
    bits = _bf16_bits(t).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def tolerance(c: int, r: int, s: int) -> Tuple[float, float]:
    """(rtol, atol) of the parity bar: |gpu - ref| <= 1e-5*|ref| + 1e-4*sqrt(C*R*S).

    For a grouped convolution pass the channels one output sums over, C/groups."""
    return 1e-5, 1e-4 * float(np.sqrt(c * r * s))
