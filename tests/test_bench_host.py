"""Host-side pieces of the benchmark (CPU only): the algorithmic byte counts of every
line it can print, the output-gradient generator, and the reference arm's JSON line."""
import json
import math
import os
import subprocess
import sys

import pytest

import bench
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_gradient_and_bf16_byte_counts():
    wl = workloads.get("resnet_28x28_c256")  # stride 1, pad 1: every input pixel is touched
    p, q = bench.shape_of(wl)
    x_b = wl.n * wl.h * wl.w * wl.c * 2
    w_b = wl.k * wl.r * wl.s * wl.c * 2
    assert bench.algorithmic_bytes(wl, 2) == x_b + w_b + wl.n * p * q * wl.k * 2 + wl.k * 4
    assert bench.algorithmic_bytes_wgrad(wl) == x_b + wl.n * p * q * wl.k * 2 + wl.k * wl.r * wl.s * wl.c * 4
    assert bench.algorithmic_bytes_dgrad(wl) == wl.n * p * q * wl.k * 2 + w_b + x_b * 2


def test_output_gradient_generator():
    wl = workloads.get("resnet_56x56_c64")
    dy = workloads.make_output_grad(wl)
    assert tuple(dy.shape) == (4, 56, 56, 64) and str(dy.dtype) == "torch.bfloat16"
    L = 4 * 56 * 56
    var = float(dy.float().var())
    assert abs(var / (2.0 / L) - 1.0) < 0.05
    unit = workloads.make_output_grad(wl, variance=1.0)
    assert abs(float(unit.float().var()) - 1.0) < 0.05
    assert workloads.make_output_grad(wl).equal(dy)  # seeded


@pytest.mark.parametrize("op", ["fwd", "wgrad", "dgrad"])
def test_reference_arm_prints_one_json_line(op):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--op", op, "--workload",
           "tiny_8x8_c16" if op == "fwd" else "resnet_56x56_c64", "--steps", "2", "--warmup", "1"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT,
                         env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "gpu_launches"):
        assert key in d, key
    assert d["impl"] == "reference" and d["gpu_launches"] == 0 and d["value"] > 0 and math.isfinite(d["value"])
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert ("wgrad" in d["metric"]) == (op == "wgrad") and ("dgrad" in d["metric"]) == (op == "dgrad")


def test_traffic_table_format_and_hash_gate(monkeypatch):
    """profiles/ncu_traffic.txt: one line per workload (optionally :wgrad / :dgrad) with the kernel
    sources' hash and a positive byte count; the bench reports a figure only while the hash matches."""
    lines = [l.split() for l in open(os.path.join(ROOT, "profiles", "ncu_traffic.txt")).read().splitlines()
             if l.strip() and not l.startswith("#")]
    assert lines
    hashes = set()
    for name, h, nbytes in lines:
        wl_name, _, op = name.partition(":")
        assert wl_name in workloads.WORKLOADS and op in ("", "wgrad", "dgrad"), name
        assert len(h) == 16 and int(h, 16) >= 0
        assert int(nbytes) > 0
        hashes.add(h)
    assert len(hashes) == 1  # one capture of one source tree
    table_hash = hashes.pop()
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: table_hash)
    want = {name: float(nbytes) for name, _, nbytes in lines}
    assert bench.recorded_traffic("resnet_28x28_c256") == want["resnet_28x28_c256"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.recorded_traffic("resnet_28x28_c256") is None
