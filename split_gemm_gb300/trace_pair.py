"""Per-stage timeline of the CTA-pair kernels (a profiling tool, not part of the call path).

Builds a second copy of the library with the trace hooks compiled in (`-DSGB_TRACE_ENABLED`:
`SGB_TRACE`, `SGB_TRACE_VALUE` and `SGB_PAIR_MARK` in `csrc/trace.cuh` write global-timer
stamps and SM-cycle counts into a device buffer), runs one workload a few times with the
heuristic's or a forced plan, and prints for the first CTAs their dependency release,
accumulator-ready and epilogue-done times, the epilogue's per-slab SM-cycle stamps, and for
pair 0 every pipeline stage's load issue, landing, MMA start and MMA issue end.

    python -m split_gemm_gb300.trace_pair --workload resnet_28x28_c256 [--loader 10 --grid 56 --block-n 256]

Reading the numbers: a global-timer read costs a few tens of nanoseconds and the trace
stores go to global memory, so intervals of a few hundred nanoseconds or less are only
indicative; the copy traced is the same kernel code with the hooks in.
"""
import argparse
import concurrent.futures as cf
import ctypes
import os
import subprocess
import sys

from . import _build

TRACE_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib_trace")
TRACE_LIB = os.path.join(TRACE_DIR, "libconv2d_trace.so")
TRACE_WORDS = 8192 + 8 * 256  # 32 slots per CTA for 256 CTAs, then 256 stages x 8 events of pair 0


def build_trace_library() -> str:
    """Compile the library's sources with the trace hooks into a separate shared object."""
    os.makedirs(TRACE_DIR, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(TRACE_DIR, os.path.splitext(src)[0] + ".o")
        cmd = [_build.nvcc(), *_build.ARCH, *_build.NVCC_FLAGS, "-DSGB_TRACE_ENABLED", "-c",
               os.path.join(_build.CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode:
            raise RuntimeError(f"nvcc failed for {src}:\n{res.stderr}")
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(_build.SOURCES)) as ex:
        objs = list(ex.map(compile_one, _build.SOURCES))
    res = subprocess.run([_build.nvcc(), *_build.ARCH, "-shared", "-o", TRACE_LIB, *objs], capture_output=True,
                         text=True)
    if res.returncode:
        raise RuntimeError(f"link failed:\n{res.stderr}")
    return TRACE_LIB


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--workload", default="resnet_28x28_c256")
    ap.add_argument("--loader", type=int, default=0)
    ap.add_argument("--grid", type=int, default=0)
    ap.add_argument("--block-n", type=int, default=0)
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--ctas", type=int, default=4, help="CTAs whose phases are printed")
    ap.add_argument("--no-build", action="store_true", help="reuse the trace library already built")
    a = ap.parse_args(argv)

    import torch
    import split_gemm_gb300 as sg
    sys.path.insert(0, _build.ROOT)
    import workloads

    lib_path = TRACE_LIB if a.no_build else build_trace_library()
    lib = sg._bind(ctypes.CDLL(lib_path))
    lib.conv2d_debug_set_trace.argtypes = [ctypes.c_void_p]
    sg._lib = lib  # this process's calls go to the traced copy

    dev = torch.device("cuda", 0)
    wl = workloads.get(a.workload)
    x, w, b = workloads.make_inputs(wl)
    xd, wd = x.to(dev), w.to(dev)
    bd = None if b is None else b.to(dev)
    params = sg.make_params(x.shape, w.shape, **wl.options())
    p, q = sg.output_shape(params)
    y = torch.empty((wl.n, p, q, wl.k), dtype=torch.float32, device=dev)
    ws = torch.zeros(max(4096, sg.workspace_bytes(params)), dtype=torch.uint8, device=dev)
    algo = None
    if a.loader or a.grid or a.block_n or a.splits:
        algo = sg.Algo()
        algo.loader, algo.grid, algo.block_n, algo.splits = a.loader, a.grid, a.block_n, a.splits
    trace = torch.zeros(TRACE_WORDS, dtype=torch.int64, device=dev)
    lib.conv2d_debug_set_trace(ctypes.c_void_p(trace.data_ptr()))
    for _ in range(3):  # the last launch is the one printed (the first ones warm caches and clocks)
        trace.zero_()
        sg.conv2d_fwd_into(y, xd, wd, bd, **wl.options(), workspace=ws, algo=algo)
        torch.cuda.synchronize()
    lib.conv2d_debug_set_trace(None)
    t = trace.cpu().tolist()
    t0 = t[1]

    def rel(v):
        return v - t0 if v else -1

    print(f"{wl.name}: times in ns after CTA 0's dependency release")
    for cta in range(a.ctas):
        row = t[cta * 32: cta * 32 + 32]
        if row[0] == 0:
            continue
        print(f" cta {cta}: start {rel(row[0])} release {rel(row[1])} seg0 ready {rel(row[2])} done {rel(row[3])}"
              f" seg1 ready {rel(row[4])} done {rel(row[5])} exit {rel(row[10])}")
        for seg in range(2):
            cyc = row[12 + 8 * seg: 20 + 8 * seg]
            if any(cyc):
                print(f"   seg{seg} epilogue SM cycles after the grant, (slab in registers, slab stored) x 4: {cyc}")
    print(" stage: activation issue (leader, peer)  landed  MMA start  MMA issue end  weight issue (leader, peer)")
    for i in range(200):
        e = t[8192 + 8 * i: 8192 + 8 * i + 7]
        if e[3] == 0:
            break
        print(f"  {i:3d}: {rel(e[0]):7d} {rel(e[1]):7d} {rel(e[2]):7d} {rel(e[3]):7d} {rel(e[4]):7d}"
              f" {rel(e[5]):7d} {rel(e[6]):7d}")
    halo = [(rel(t[8192 + 8 * (200 + h)]), rel(t[8192 + 8 * (200 + h) + 1])) for h in range(8)
            if t[8192 + 8 * (200 + h)]]
    if halo:
        print(" halo issues (leader, peer):", halo)
    return 0


if __name__ == "__main__":
    sys.exit(main())
