"""The C ABI library loads and exports what include/*.h declares; host-only calls (no GPU)."""
import ctypes
import glob
import os
import re

import pytest

import split_gemm_gb300 as sg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(hdr).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([a-z_][a-z0-9_]*)\s*\(", text, re.M):
            names.append(m.group(1))
    return sorted(set(names))


def test_header_declares_the_binding_symbols():
    assert set(declared_functions()) == set(sg.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(sg.load_library()._name)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def _params(**kw):
    base = dict(x_shape=(4, 56, 56, 64), w_shape=(64, 3, 3, 64), stride=1, padding=1, dilation=1)
    base.update(kw)
    return sg.make_params(base["x_shape"], base["w_shape"], base["stride"], base["padding"], base["dilation"],
                          base.get("groups", 1))


def test_output_shape_host_only():
    assert sg.output_shape(_params()) == (56, 56)
    assert sg.output_shape(_params(x_shape=(32, 224, 224, 3), w_shape=(64, 7, 7, 3), stride=2, padding=3)) == (112, 112)
    assert sg.output_shape(_params(x_shape=(8, 64, 64, 128), w_shape=(128, 3, 3, 128), padding=2, dilation=2)) == (64, 64)
    assert sg.output_shape(_params(x_shape=(32, 56, 56, 256), w_shape=(512, 1, 1, 256), stride=2, padding=0)) == (28, 28)
    # grouped: the weight holds C/groups channels per tap
    assert sg.output_shape(_params(w_shape=(64, 3, 3, 16), groups=4)) == (56, 56)
    with pytest.raises(ValueError):
        _params(w_shape=(64, 3, 3, 64), groups=4)


@pytest.mark.parametrize("kw,code", [
    (dict(groups=3), 1),                                          # groups must divide C (64) and K
    (dict(groups=0), 1),
    (dict(x_shape=(1, 2, 2, 3), w_shape=(4, 5, 5, 3), padding=0), 1),  # window does not fit
    (dict(stride=0), 1),
    (dict(dilation=0), 1),
    (dict(padding=-1), 1),
])
def test_invalid_params_rejected(kw, code):
    with pytest.raises(sg.Conv2dError) as e:
        sg.output_shape(_params(**kw))
    assert e.value.code == code


def test_workspace_and_staging_sizes():
    p = _params()
    # status block + one semaphore per 128 x 64 tile of the finest tiling any loader can be forced to
    # use: the halo loader's 128-pixel tiles of each image seen with the padded row pitch 58 (26 per
    # image, 4 images)
    assert sg.workspace_bytes(p) == 256 + 4 * 26 * 1 * 4
    assert sg.host_staging_bytes(p) >= (4 * 56 * 56 * 64 * 2 + 64 * 576 * 2 + 12544 * 64 * 4)


def test_strerror_covers_codes():
    for code in range(8):
        assert sg.strerror(code)
    assert sg.strerror(99) == "unknown status"


@pytest.mark.parametrize("act,dtype", [(2, 0), (-1, 0), (0, 2), (1, -3)])
def test_unknown_epilogue_rejected_before_any_device_work(act, dtype):
    """An unknown activation or output type is CONV2D_ERR_INVALID; the check runs on the host
    before anything touches the (here fake, never dereferenced) device pointers."""
    lib = sg.load_library()
    p = _params()
    fake = 1 << 20  # 16-byte aligned, non-null
    rc = lib.conv2d_fwd_epi(ctypes.byref(p), fake, fake, None, fake, None, 0, None, None,
                            ctypes.byref(sg.Epilogue(act, dtype)))
    assert rc == 1
