"""The product path has no CPU fallback (CPU only): a missing library is an error, and the
binding refuses host tensors instead of computing anything on the CPU."""
import subprocess
import sys

import pytest
import torch

import split_gemm_gb300 as sg


def test_missing_library_raises():
    code = (
        "import split_gemm_gb300 as sg, split_gemm_gb300._build as b\n"
        "b.LIB_PATH = '/nonexistent/libconv2d.so'\n"
        "try:\n"
        "    sg.load_library(build_if_stale=False)\n"
        "except RuntimeError as e:\n"
        "    print('raised', 'missing' in str(e))\n"
    )
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert res.stdout.strip() == "raised True", res.stdout + res.stderr


def _bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


@pytest.mark.parametrize("call", [
    lambda: sg.conv2d_fwd(_bf16(1, 8, 8, 64), _bf16(64, 3, 3, 64), padding=1),
    lambda: sg.conv2d_fwd(_bf16(1, 8, 8, 64), _bf16(64, 3, 3, 64), padding=1, relu=True, out_dtype=torch.bfloat16),
    lambda: sg.conv2d_bwd_weight(_bf16(1, 8, 8, 64), _bf16(1, 8, 8, 64), (64, 3, 3, 64), padding=1),
    lambda: sg.conv2d_bwd_data(_bf16(1, 8, 8, 64), _bf16(64, 3, 3, 64), (1, 8, 8, 64), padding=1),
    lambda: sg.conv_transpose2d(_bf16(1, 8, 8, 64), _bf16(64, 3, 3, 64), padding=1),
], ids=["fwd", "fwd_fused", "wgrad", "dgrad", "conv_transpose2d"])
def test_host_tensors_are_refused(call):
    with pytest.raises(ValueError, match="CUDA tensor"):
        call()
