"""Build the CUDA library libmoe_b300.so in-tree (nvcc, sm_103a only).

    python -m mixture_experts_layer_87_b300.build [--force] [--check] [-v]

--check builds the range-checked variant libmoe_b300_check.so (-DMOE_CHECK:
every computed index of a global access is checked against its buffer and
an out-of-range one is recorded in the status word and skipped; see
MOE_IN_RANGE in csrc/ptx.cuh).  The binding loads it instead of the normal
library when MOE_B300_LIBRARY=check is set.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
SO = os.path.join(PKG, "libmoe_b300.so")
SO_CHECK = os.path.join(PKG, "libmoe_b300_check.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
]


def sources():
    srcs = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC)) if f.endswith((".cu", ".cuh"))]
    return srcs + [os.path.join(INCLUDE, "moe.h")]


def needs_build(so: str = SO) -> bool:
    if not os.path.exists(so):
        return True
    t = os.path.getmtime(so)
    return any(os.path.getmtime(s) > t for s in sources())


def build(force: bool = False, verbose: bool = False, check: bool = False) -> str:
    so = SO_CHECK if check else SO
    if not force and not needs_build(so):
        return so
    nvcc = os.environ.get("NVCC", "nvcc")
    cmd = [nvcc, *NVCC_FLAGS, *(["-DMOE_CHECK"] if check else []), "-I" + INCLUDE, "-I" + CSRC,
           os.path.join(CSRC, "moe_api.cu"), "-o", so + ".tmp"]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.check_call(cmd)
    os.replace(so + ".tmp", so)
    return so


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, check="--check" in sys.argv))
