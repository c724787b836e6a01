"""Build the CUDA libraries in-tree with nvcc for sm_103a: libbitlinear.so (the
C-ABI BitLinear library, every .cu under csrc/) and libbitlinear_probe.so (the
tensor-core peak microbenchmarks under csrc/probe/, used by bench.py only)."""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libbitlinear.so")
PROBE_LIB = os.path.join(HERE, "libbitlinear_probe.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def probe_sources():
    return sorted(glob.glob(os.path.join(CSRC, "probe", "*.cu")))


def _stale(lib: str, srcs) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = list(srcs) + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        [os.path.join(os.path.dirname(HERE), "include", "bitlinear.h")]
    return any(os.path.getmtime(p) > t for p in deps)


def _link(lib: str, srcs, objdir: str, verbose: bool) -> None:
    os.makedirs(objdir, exist_ok=True)
    objs = []
    for src in srcs:
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        cmd = [NVCC, *ARCH, *FLAGS, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        subprocess.check_call(cmd)
        objs.append(obj)
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.check_call([NVCC, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, lib)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile both libraries (when stale); returns the path of libbitlinear.so."""
    if force or _stale(LIB, sources()):
        _link(LIB, sources(), os.path.join(HERE, "_build"), verbose)
    if force or _stale(PROBE_LIB, probe_sources()):
        _link(PROBE_LIB, probe_sources(), os.path.join(HERE, "_build", "probe"), verbose)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
