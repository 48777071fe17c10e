"""GB300 (sm_103a) implicit-GEMM 2-D convolution forward: Python binding.

This module only marshals arguments to the C ABI in ``include/conv2d.h``
(``libconv2d.so``, built in-tree by ``split_gemm_gb300._build``).  Every step of
the computation runs in the library's CUDA kernels; PyTorch provides device
memory and the current stream.  There is no fallback: if the library cannot be
loaded, every call raises.

    y = conv2d_fwd(x, w, bias, stride=1, padding=0, dilation=1)
      x: [N,H,W,C] bf16 CUDA tensor (NHWC), w: [K,R,S,C] bf16 (KRSC),
      bias: [K] fp32 or None  ->  y: [N,P,Q,K] fp32 (NHWC)

    y = conv2d_fwd(x, w, bias, relu=True, out_dtype=torch.bfloat16)
      the fused epilogue: ReLU after the bias, y stored as bf16 (whole-tile plans)
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

from . import _build

__all__ = [
    "Conv2dError", "Params", "Algo", "LOADER_AUTO", "LOADER_TMA_IM2COL", "LOADER_CPASYNC", "LOADER_SCALAR",
    "LOADER_HYBRID", "LOADER_ROW_WINDOW", "LOADER_TMA_BOX", "LOADER_HALO", "LOADER_DIRECT", "LOADER_TMA_PAIR", "LOADER_PAIR_HALO", "LOADER_BLOCKDIAG", "REDUCTION_AUTO", "REDUCTION_ORDERED",
    "REDUCTION_CONCURRENT", "Epilogue", "ACT_NONE", "ACT_RELU", "OUT_F32", "OUT_BF16",
    "DEBUG_SKIP_SIGNAL", "DEBUG_TMA_STORE", "load_library", "library_path", "make_params", "output_shape", "workspace_bytes",
    "query_algo", "epi_workspace_bytes", "conv2d_bwd_weight", "conv2d_bwd_weight_into",
    "wgrad_workspace_bytes", "query_wgrad_algo", "conv2d_bwd_data", "conv2d_bwd_data_into", "dgrad_workspace_bytes",
    "query_dgrad_algo", "conv_transpose2d", "conv2d_fwd", "conv2d_fwd_into", "conv2d_fwd_host", "host_staging_bytes", "status",
    "last_launch_count", "strerror", "EXPORTED_SYMBOLS", "tensor_map_cache_stats",
]

LOADER_AUTO, LOADER_TMA_IM2COL, LOADER_CPASYNC, LOADER_SCALAR, LOADER_HYBRID, LOADER_ROW_WINDOW = 0, 1, 2, 3, 4, 5
LOADER_TMA_BOX = 6
LOADER_HALO = 7
LOADER_DIRECT = 8
LOADER_TMA_PAIR = 9
LOADER_PAIR_HALO = 10
LOADER_BLOCKDIAG = 11
REDUCTION_AUTO, REDUCTION_ORDERED, REDUCTION_CONCURRENT = 0, 1, 2
ACT_NONE, ACT_RELU = 0, 1
OUT_F32, OUT_BF16 = 0, 1
DEBUG_SKIP_SIGNAL = 1
DEBUG_TMA_STORE = 8  # CTA-pair loaders: write y through TMA stores (measurement hook; slower)
STATUS_NAMES = {0: "CONV2D_OK", 1: "CONV2D_ERR_INVALID", 2: "CONV2D_ERR_UNSUPPORTED", 3: "CONV2D_ERR_ALIGNMENT",
                4: "CONV2D_ERR_WORKSPACE", 5: "CONV2D_ERR_CUDA", 6: "CONV2D_ERR_TIMEOUT",
                7: "CONV2D_ERR_SCRATCH_LIMIT"}

EXPORTED_SYMBOLS = [
    "conv2d_fwd_output_shape", "conv2d_fwd_workspace_bytes", "conv2d_fwd", "conv2d_fwd_ex",
    "conv2d_fwd_query_algo", "conv2d_fwd_status", "conv2d_fwd_host_staging_bytes", "conv2d_fwd_host",
    "conv2d_last_launch_count", "conv2d_strerror", "conv2d_fwd_noalloc", "conv2d_fwd_epi",
    "conv2d_tensor_map_cache_stats",
    "conv2d_fwd_query_algo_epi", "conv2d_fwd_epi_workspace_bytes", "conv2d_bwd_weight_workspace_bytes",
    "conv2d_bwd_weight", "conv2d_bwd_weight_query_algo", "conv2d_bwd_data_workspace_bytes", "conv2d_bwd_data",
    "conv2d_bwd_data_query_algo",
]


class Conv2dError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({_strerror_or_code(code)})")


class Params(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int64), ("h", ctypes.c_int64), ("w", ctypes.c_int64), ("c", ctypes.c_int64),
                ("k", ctypes.c_int64), ("r", ctypes.c_int64), ("s", ctypes.c_int64),
                ("stride_h", ctypes.c_int32), ("stride_w", ctypes.c_int32),
                ("pad_h", ctypes.c_int32), ("pad_w", ctypes.c_int32),
                ("dil_h", ctypes.c_int32), ("dil_w", ctypes.c_int32), ("groups", ctypes.c_int32)]


class Algo(ctypes.Structure):
    _fields_ = [("block_n", ctypes.c_int32), ("splits", ctypes.c_int32), ("loader", ctypes.c_int32),
                ("grid", ctypes.c_int32), ("debug_flags", ctypes.c_int32), ("block_m", ctypes.c_int32),
                ("wait_limit_ns", ctypes.c_int64), ("reduction", ctypes.c_int32)]

    def as_dict(self):
        return dict(block_m=self.block_m, block_n=self.block_n, splits=self.splits, loader=self.loader,
                    grid=self.grid, reduction=self.reduction)


class Epilogue(ctypes.Structure):
    _fields_ = [("activation", ctypes.c_int32), ("out_dtype", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def _bind(lib):
    P = ctypes.POINTER(Params)
    A = ctypes.POINTER(Algo)
    vp, sz, i64p = ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(ctypes.c_int64)
    lib.conv2d_fwd_output_shape.argtypes = [P, i64p, i64p]
    lib.conv2d_fwd_output_shape.restype = ctypes.c_int
    lib.conv2d_fwd_workspace_bytes.argtypes = [P]
    lib.conv2d_fwd_workspace_bytes.restype = sz
    lib.conv2d_fwd.argtypes = [P, vp, vp, vp, vp, vp, sz, vp]
    lib.conv2d_fwd.restype = ctypes.c_int
    lib.conv2d_fwd_ex.argtypes = [P, vp, vp, vp, vp, vp, sz, vp, A]
    lib.conv2d_fwd_ex.restype = ctypes.c_int
    lib.conv2d_fwd_epi.argtypes = [P, vp, vp, vp, vp, vp, sz, vp, A, ctypes.POINTER(Epilogue)]
    lib.conv2d_fwd_epi.restype = ctypes.c_int
    lib.conv2d_fwd_epi_workspace_bytes.argtypes = [P, A, ctypes.POINTER(Epilogue)]
    lib.conv2d_fwd_epi_workspace_bytes.restype = sz
    lib.conv2d_fwd_query_algo_epi.argtypes = [P, ctypes.POINTER(Epilogue), A]
    lib.conv2d_fwd_query_algo_epi.restype = ctypes.c_int
    lib.conv2d_bwd_data_workspace_bytes.argtypes = [P]
    lib.conv2d_bwd_data_workspace_bytes.restype = sz
    lib.conv2d_bwd_data.argtypes = [P, vp, vp, vp, vp, sz, vp, A]
    lib.conv2d_bwd_data.restype = ctypes.c_int
    lib.conv2d_bwd_data_query_algo.argtypes = [P, A]
    lib.conv2d_bwd_data_query_algo.restype = ctypes.c_int
    lib.conv2d_bwd_weight_workspace_bytes.argtypes = [P]
    lib.conv2d_bwd_weight_workspace_bytes.restype = sz
    lib.conv2d_bwd_weight.argtypes = [P, vp, vp, vp, vp, sz, vp, A]
    lib.conv2d_bwd_weight.restype = ctypes.c_int
    lib.conv2d_bwd_weight_query_algo.argtypes = [P, A]
    lib.conv2d_bwd_weight_query_algo.restype = ctypes.c_int
    lib.conv2d_fwd_query_algo.argtypes = [P, A]
    lib.conv2d_fwd_query_algo.restype = ctypes.c_int
    lib.conv2d_fwd_status.argtypes = [vp, sz, vp]
    lib.conv2d_fwd_status.restype = ctypes.c_int
    lib.conv2d_fwd_host_staging_bytes.argtypes = [P]
    lib.conv2d_fwd_host_staging_bytes.restype = sz
    lib.conv2d_fwd_host.argtypes = [P, vp, vp, vp, vp, vp, sz, vp]
    lib.conv2d_fwd_host.restype = ctypes.c_int
    lib.conv2d_last_launch_count.argtypes = []
    lib.conv2d_last_launch_count.restype = ctypes.c_int
    lib.conv2d_tensor_map_cache_stats.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), ctypes.POINTER(ctypes.c_ulonglong)]
    lib.conv2d_tensor_map_cache_stats.restype = None
    lib.conv2d_fwd_noalloc.argtypes = [P, vp, vp, vp, vp, vp]
    lib.conv2d_fwd_noalloc.restype = ctypes.c_int
    lib.conv2d_strerror.argtypes = [ctypes.c_int]
    lib.conv2d_strerror.restype = ctypes.c_char_p
    return lib


def load_library(build_if_stale: bool = True):
    """Load (building first if needed) the CUDA library; raises if that is impossible."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if build_if_stale and not _build.up_to_date():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"split_gemm_gb300: CUDA library {path} is missing; run __graft_entry__.build()")
        _lib = _bind(ctypes.CDLL(path))
        return _lib


def _strerror_or_code(code: int) -> str:
    try:
        return load_library(build_if_stale=False).conv2d_strerror(code).decode()
    except Exception:  # the message is best effort; the code is in the exception
        return str(code)


def strerror(code: int) -> str:
    return load_library().conv2d_strerror(code).decode()


def _pair(v) -> Tuple[int, int]:
    if isinstance(v, (tuple, list)):
        return int(v[0]), int(v[1])
    return int(v), int(v)


def make_params(x_shape, w_shape, stride=1, padding=0, dilation=1, groups=1) -> Params:
    n, h, w, c = (int(v) for v in x_shape)
    k, r, s, c2 = (int(v) for v in w_shape)
    # The weight holds C/groups channels per tap; whether `groups` itself is valid
    # (>= 1, dividing C and K) is the C ABI's call.
    if int(groups) >= 1 and c % int(groups) == 0 and c2 * int(groups) != c:
        raise ValueError(f"channel mismatch: input C={c}, weight C/groups={c2}, groups={groups}")
    sh, sw = _pair(stride)
    ph, pw = _pair(padding)
    dh, dw = _pair(dilation)
    return Params(n, h, w, c, k, r, s, sh, sw, ph, pw, dh, dw, int(groups))


def output_shape(params: Params) -> Tuple[int, int]:
    p, q = ctypes.c_int64(), ctypes.c_int64()
    rc = load_library().conv2d_fwd_output_shape(ctypes.byref(params), ctypes.byref(p), ctypes.byref(q))
    if rc:
        raise Conv2dError(rc, "conv2d_fwd_output_shape")
    return p.value, q.value


def workspace_bytes(params: Params) -> int:
    return int(load_library().conv2d_fwd_workspace_bytes(ctypes.byref(params)))


def epi_workspace_bytes(params: Params, algo: Optional[Algo] = None, relu: bool = False,
                        out_bf16: bool = False) -> int:
    """Workspace bytes a fused-epilogue call needs with this configuration (None: the heuristic's)."""
    epi = Epilogue(ACT_RELU if relu else ACT_NONE, OUT_BF16 if out_bf16 else OUT_F32)
    return int(load_library().conv2d_fwd_epi_workspace_bytes(
        ctypes.byref(params), None if algo is None else ctypes.byref(algo), ctypes.byref(epi)))


def host_staging_bytes(params: Params) -> int:
    return int(load_library().conv2d_fwd_host_staging_bytes(ctypes.byref(params)))


def query_algo(params: Params, relu: bool = False, out_bf16: bool = False) -> Algo:
    """The heuristic's configuration; with ``relu``/``out_bf16`` that of the fused epilogue's call."""
    out = Algo()
    if relu or out_bf16:
        epi = Epilogue(ACT_RELU if relu else ACT_NONE, OUT_BF16 if out_bf16 else OUT_F32)
        rc = load_library().conv2d_fwd_query_algo_epi(ctypes.byref(params), ctypes.byref(epi), ctypes.byref(out))
    else:
        rc = load_library().conv2d_fwd_query_algo(ctypes.byref(params), ctypes.byref(out))
    if rc:
        raise Conv2dError(rc, "conv2d_fwd_query_algo")
    return out


def last_launch_count() -> int:
    return int(load_library().conv2d_last_launch_count())


def tensor_map_cache_stats():
    """(hits, misses) of the forward calls' tensor-map cache since the library was loaded."""
    h, m = ctypes.c_ulonglong(0), ctypes.c_ulonglong(0)
    load_library().conv2d_tensor_map_cache_stats(ctypes.byref(h), ctypes.byref(m))
    return int(h.value), int(m.value)


# Per-device zero-filled workspaces (the kernels leave them zeroed after each call).
# They assume one stream at a time per device; pass `workspace=` for concurrent streams.
_ws_cache = {}


def _default_workspace(nbytes: int, device):
    import torch
    key = device.index if device.index is not None else torch.cuda.current_device()
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.zeros(max(nbytes, 4096), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def _mark_used(buf, stream) -> None:
    """Tells torch's caching allocator that the cached workspace ``buf`` is in use by
    ``stream``: if a later, larger call replaces it, its memory is not handed out again
    until the work already queued on that stream has finished."""
    if stream is not None and buf.device.type == "cuda":
        buf.record_stream(stream)


def _check_tensor(t, name, dtype, ndim):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def conv2d_fwd_into(y, x, w, bias=None, stride=1, padding=0, dilation=1, groups=1, *, workspace=None,
                    algo: Optional[Algo] = None, stream=None, relu: bool = False) -> None:
    """Writes conv2d(x, w) + bias into the preallocated NHWC tensor ``y`` (asynchronous).

    ``y`` is fp32, or bf16 for the fused bf16-output epilogue; ``relu`` applies
    max(v, 0) after the bias.  Under either fused option a tile cut between CTAs is
    summed in an fp32 buffer in the workspace and finished by its last CTA.
    """
    import torch
    _check_tensor(x, "x", torch.bfloat16, 4)
    _check_tensor(w, "w", torch.bfloat16, 4)
    _check_tensor(y, "y", torch.bfloat16 if y.dtype == torch.bfloat16 else torch.float32, 4)
    if bias is not None:
        _check_tensor(bias, "bias", torch.float32, 1)
    params = make_params(x.shape, w.shape, stride, padding, dilation, groups)
    lib = load_library()
    fused = relu or y.dtype == torch.bfloat16
    cached = workspace is None
    if workspace is None:
        need = workspace_bytes(params)
        # A fused call whose plan cuts tiles also needs the fp32 partial-sum buffer (the direct
        # kernel for small groups, which the heuristic picks when nothing is forced, needs none).
        if fused and not (algo is None and query_algo(params).loader == LOADER_DIRECT):
            need = epi_workspace_bytes(params, algo, relu, y.dtype == torch.bfloat16)
        workspace = _default_workspace(need, x.device)
    ws_ptr, ws_len = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = torch.cuda.current_stream(x.device) if stream is None else stream
    args = (ctypes.byref(params), x.data_ptr(), w.data_ptr(), None if bias is None else bias.data_ptr(),
            y.data_ptr(), ws_ptr, ws_len, st.cuda_stream)
    if fused:
        epi = Epilogue(ACT_RELU if relu else ACT_NONE, OUT_BF16 if y.dtype == torch.bfloat16 else OUT_F32)
        rc = lib.conv2d_fwd_epi(*args, None if algo is None else ctypes.byref(algo), ctypes.byref(epi))
    else:
        rc = lib.conv2d_fwd(*args) if algo is None else lib.conv2d_fwd_ex(*args, ctypes.byref(algo))
    if rc:
        raise Conv2dError(rc, "conv2d_fwd")
    if cached:
        _mark_used(workspace, st)


def conv2d_fwd(x, w, bias=None, stride=1, padding=0, dilation=1, groups=1, *, workspace=None,
               algo: Optional[Algo] = None, stream=None, relu: bool = False, out_dtype=None):
    """Returns y = conv2d(x, w) + bias as a new NHWC CUDA tensor (asynchronous).

    ``out_dtype``: torch.float32 (default) or torch.bfloat16; ``relu``: see conv2d_fwd_into.
    """
    import torch
    out_dtype = torch.float32 if out_dtype is None else out_dtype
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise TypeError(f"out_dtype must be torch.float32 or torch.bfloat16, got {out_dtype}")
    params = make_params(x.shape, w.shape, stride, padding, dilation, groups)
    p, q = output_shape(params)
    y = torch.empty((params.n, p, q, params.k), dtype=out_dtype, device=x.device)
    conv2d_fwd_into(y, x, w, bias, stride, padding, dilation, groups, workspace=workspace, algo=algo,
                    stream=stream, relu=relu)
    return y


def wgrad_workspace_bytes(params: Params) -> int:
    return int(load_library().conv2d_bwd_weight_workspace_bytes(ctypes.byref(params)))


def query_wgrad_algo(params: Params) -> Algo:
    """The heuristic's configuration for the weight gradient of this convolution."""
    out = Algo()
    rc = load_library().conv2d_bwd_weight_query_algo(ctypes.byref(params), ctypes.byref(out))
    if rc:
        raise Conv2dError(rc, "conv2d_bwd_weight_query_algo")
    return out


def conv2d_bwd_weight_into(dw, x, dy, stride=1, padding=0, dilation=1, groups=1, *, workspace=None,
                           algo: Optional[Algo] = None, stream=None) -> None:
    """Writes the weight gradient of conv2d(x, w) for output gradient ``dy`` into the fp32
    tensor ``dw`` [K,R,S,C] (asynchronous).  x [N,H,W,C] and dy [N,P,Q,K] are bf16 CUDA tensors."""
    import torch
    _check_tensor(x, "x", torch.bfloat16, 4)
    _check_tensor(dy, "dy", torch.bfloat16, 4)
    _check_tensor(dw, "dw", torch.float32, 4)
    params = make_params(x.shape, dw.shape, stride, padding, dilation, groups)
    p, q = output_shape(params)
    if tuple(dy.shape) != (params.n, p, q, params.k):
        raise ValueError(f"dy must be [{params.n}, {p}, {q}, {params.k}], got {list(dy.shape)}")
    lib = load_library()
    cached = workspace is None
    if workspace is None:
        workspace = _default_workspace(wgrad_workspace_bytes(params), x.device)
    st = torch.cuda.current_stream(x.device) if stream is None else stream
    rc = lib.conv2d_bwd_weight(ctypes.byref(params), x.data_ptr(), dy.data_ptr(), dw.data_ptr(), workspace.data_ptr(),
                               workspace.numel() * workspace.element_size(), st.cuda_stream,
                               None if algo is None else ctypes.byref(algo))
    if rc:
        raise Conv2dError(rc, "conv2d_bwd_weight")
    if cached:
        _mark_used(workspace, st)


def conv2d_bwd_weight(x, dy, w_shape, stride=1, padding=0, dilation=1, groups=1, *, workspace=None,
                      algo: Optional[Algo] = None, stream=None):
    """Returns the weight gradient [K,R,S,C/groups] fp32 as a new CUDA tensor (asynchronous)."""
    import torch
    dw = torch.empty(tuple(int(v) for v in w_shape), dtype=torch.float32, device=x.device)
    conv2d_bwd_weight_into(dw, x, dy, stride, padding, dilation, groups, workspace=workspace, algo=algo,
                           stream=stream)
    return dw


def dgrad_workspace_bytes(params: Params) -> int:
    return int(load_library().conv2d_bwd_data_workspace_bytes(ctypes.byref(params)))


def query_dgrad_algo(params: Params) -> Algo:
    """The heuristic's configuration for the data gradient of this convolution."""
    out = Algo()
    rc = load_library().conv2d_bwd_data_query_algo(ctypes.byref(params), ctypes.byref(out))
    if rc:
        raise Conv2dError(rc, "conv2d_bwd_data_query_algo")
    return out


def conv2d_bwd_data_into(dx, dy, w, stride=1, padding=0, dilation=1, groups=1, *, workspace=None,
                         algo: Optional[Algo] = None, stream=None) -> None:
    """Writes the input gradient of conv2d(x, w) for output gradient ``dy`` into the fp32
    tensor ``dx`` [N,H,W,C] (asynchronous).  dy [N,P,Q,K] and w [K,R,S,C] are bf16 CUDA tensors."""
    import torch
    _check_tensor(dy, "dy", torch.bfloat16, 4)
    _check_tensor(w, "w", torch.bfloat16, 4)
    _check_tensor(dx, "dx", torch.float32, 4)
    params = make_params(dx.shape, w.shape, stride, padding, dilation, groups)
    p, q = output_shape(params)
    if tuple(dy.shape) != (params.n, p, q, params.k):
        raise ValueError(f"dy must be [{params.n}, {p}, {q}, {params.k}], got {list(dy.shape)}")
    lib = load_library()
    cached = workspace is None
    if workspace is None:
        workspace = _default_workspace(dgrad_workspace_bytes(params), dy.device)
    st = torch.cuda.current_stream(dy.device) if stream is None else stream
    rc = lib.conv2d_bwd_data(ctypes.byref(params), dy.data_ptr(), w.data_ptr(), dx.data_ptr(), workspace.data_ptr(),
                             workspace.numel() * workspace.element_size(), st.cuda_stream,
                             None if algo is None else ctypes.byref(algo))
    if rc:
        raise Conv2dError(rc, "conv2d_bwd_data")
    if cached:
        _mark_used(workspace, st)


def conv2d_bwd_data(dy, w, x_shape, stride=1, padding=0, dilation=1, groups=1, *, workspace=None,
                    algo: Optional[Algo] = None, stream=None):
    """Returns the input gradient [N,H,W,C] fp32 for a forward input of shape ``x_shape``."""
    import torch
    dx = torch.empty(tuple(int(v) for v in x_shape), dtype=torch.float32, device=dy.device)
    conv2d_bwd_data_into(dx, dy, w, stride, padding, dilation, groups, workspace=workspace, algo=algo, stream=stream)
    return dx


def conv_transpose2d(x, w, padding=0, dilation=1, *, stride=1, output_padding=0, workspace=None,
                     algo: Optional[Algo] = None, stream=None):
    """conv_transpose2d: x [N,Hi,Wi,Cin] bf16, w [Cin,R,S,Cout] bf16 -> y [N,Ho,Wo,Cout] fp32 with
    Ho = (Hi-1)*stride - 2*padding + dilation*(R-1) + 1 + output_padding (likewise Wo), through the
    data-gradient kernel (dy = x): the input gradient of the forward conv from Ho x Wo to Hi x Wi."""
    sh, sw = _pair(stride)
    ph, pw = _pair(padding)
    dh, dw = _pair(dilation)
    oph, opw = _pair(output_padding)
    if not (0 <= oph < sh and 0 <= opw < sw):
        raise ValueError("output_padding must lie in [0, stride)")
    n, hi, wi, cin = (int(v) for v in x.shape)
    cin_w, r, s, cout = (int(v) for v in w.shape)
    if cin_w != cin:
        raise ValueError(f"weight has {cin_w} input channels, x has {cin}")
    ho = (hi - 1) * sh - 2 * ph + dh * (r - 1) + 1 + oph
    wo = (wi - 1) * sw - 2 * pw + dw * (s - 1) + 1 + opw
    return conv2d_bwd_data(x, w, (n, ho, wo, cout), (sh, sw), (ph, pw), (dh, dw), workspace=workspace, algo=algo,
                           stream=stream)


def conv2d_fwd_host(x_host, w_host, bias_host, y_host, params: Params, staging, stream=None) -> None:
    """End-to-end call on host tensors (pinned for async copies): H2D, conv, D2H on ``stream``."""
    import torch
    st = torch.cuda.current_stream() if stream is None else stream
    rc = load_library().conv2d_fwd_host(
        ctypes.byref(params), x_host.data_ptr(), w_host.data_ptr(),
        None if bias_host is None else bias_host.data_ptr(), y_host.data_ptr(), staging.data_ptr(),
        staging.numel() * staging.element_size(), st.cuda_stream)
    if rc:
        raise Conv2dError(rc, "conv2d_fwd_host")


def status(workspace, stream=None) -> int:
    """Synchronises the stream and returns the workspace's status (0 or CONV2D_ERR_TIMEOUT)."""
    import torch
    st = torch.cuda.current_stream() if stream is None else stream
    return int(load_library().conv2d_fwd_status(workspace.data_ptr(),
                                                workspace.numel() * workspace.element_size(), st.cuda_stream))
