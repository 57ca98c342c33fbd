"""Builds libmamba_ssm.so (the C-ABI CUDA library) in-tree with nvcc, for
sm_103a only.  Usage: ``python -m selective_state_space_118_b300.build [-v]``.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libmamba_ssm.so")
SOURCES = ["kernels.cu", "api.cpp", "noalloc.cu"]
HEADERS = ["ptx.cuh", "ssm_math.cuh", "scan_fwd.cuh", "scan_bwd.cuh", "scan_complex.cuh", "step.cuh", "params.h", "launch.h", "gemm_tc.cuh", "ssd.cuh"]
PUBLIC_HEADER = os.path.join(os.path.dirname(HERE), "include", "mamba_ssm.h")

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-cudart", "shared",
         "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
LIBS = []


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [PUBLIC_HEADER, __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH, *FLAGS, "-shared", "-o", tmp]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    cmd += [os.path.join(CSRC, f) for f in SOURCES] + LIBS
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed ({r.returncode}):\n{r.stderr}")
    if verbose:
        sys.stderr.write(r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv))
