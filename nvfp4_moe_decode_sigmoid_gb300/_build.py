"""Build libflint.so in-tree: hand-written CUDA for sm_103a behind the C ABI of
include/flint.h. Translation units compile in parallel; nvcc links the CUDA
runtime statically, so the library needs only the CUDA driver (libcuda) at run time."""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libflint.so")
# The phase-trace build (FLINT_PHASE_TRACE: the fused layer kernel stamps its
# phase boundaries; used by phase_trace.py), in its own build folder.
BUILD_TRACE = os.path.join(PKG, "_build_trace")
LIB_TRACE = os.path.join(PKG, "libflint_trace.so")
SOURCES = ["abi.cu", "repack.cu", "route.cu", "gemv.cu", "layer.cu", "bf16.cu", "norm.cu", "prefill.cu"]
HEADERS = ["flint_device.cuh", "flint_internal.h", "expert_common.cuh", "router_common.cuh", "tcgen05.cuh",
           "layer_one.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "nvcc")
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall", "--expt-relaxed-constexpr",
         "-I", INCLUDE, "-I", CSRC]


def _newest_input():
    paths = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "flint.h"), __file__]
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, trace: bool = False) -> str:
    lib, bdir = (LIB_TRACE, BUILD_TRACE) if trace else (LIB, BUILD)
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input():
        return lib
    os.makedirs(bdir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(bdir, os.path.splitext(src)[0] + ".o")
        cmd = [NVCC, *ARCH, *FLAGS, *(["-DFLINT_PHASE_TRACE"] if trace else []), "-c", os.path.join(CSRC, src),
               "-o", obj]
        if os.environ.get("FLINT_PTXAS_VERBOSE"):
            cmd[1:1] = ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0 or verbose or os.environ.get("FLINT_PTXAS_VERBOSE"):
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}")
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".tmp"
    subprocess.run([NVCC, *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
