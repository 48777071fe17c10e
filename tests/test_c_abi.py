"""The C ABI from C (CPU only): include/conv2d.h compiles as C11, and a C program
linked against libconv2d.so makes the host-only calls."""
import os
import subprocess

import split_gemm_gb300 as sg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


def test_header_compiles_as_c11(tmp_path):
    src = tmp_path / "h.c"
    src.write_text('#include "conv2d.h"\nint main(void) { return (int)sizeof(conv2d_params) > 0 ? 0 : 1; }\n')
    res = subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE, "-c",
                          str(src), "-o", str(tmp_path / "h.o")], capture_output=True, text=True)
    assert res.returncode == 0, res.stderr


def test_c_program_calls_the_library(tmp_path):
    lib = sg.load_library()._name
    exe = tmp_path / "abi_host_calls"
    res = subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", INCLUDE,
                          os.path.join(ROOT, "tests", "c", "abi_host_calls.c"), lib, "-o", str(exe),
                          f"-Wl,-rpath,{os.path.dirname(lib)}"], capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60,
                         env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert run.returncode == 0, run.stdout + run.stderr
    assert "FAIL" not in run.stdout
