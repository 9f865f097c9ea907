"""Build-time resource checks of the CUDA kernels (CPU only: nvcc + ptxas -v).

* No kernel of the library spills registers to local memory.
* The FP8 expert GEMM moves registers between its warpgroups with
  setmaxnreg.  Its split (control warpgroup down, promotion warpgroups up) is
  computed from the register count that __launch_bounds__(THREADS, 1)
  allows, 65536 / THREADS rounded down to a multiple of 8. The compiled
  kernel must launch with exactly that count: with fewer, the increase could
  never be granted.  The host refuses such a build at launch time; this test
  catches it at build time.
"""
import os
import re
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from mixture_experts_layer_87_b300 import build as libbuild  # noqa: E402

ENTRY = re.compile(r"Compiling entry function '(\w+)' for 'sm_103a'")
SPILL = re.compile(r"(\d+) bytes spill stores, (\d+) bytes spill loads")
REGS = re.compile(r"Used (\d+) registers")
FP8 = re.compile(r"fp8_gemm_kernelILNS_3EpiE(\d)ELi(\d+)ELb(\d)EE")


@pytest.fixture(scope="module")
def ptxas_report(tmp_path_factory):
    nvcc = os.environ.get("NVCC", "nvcc")
    if shutil.which(nvcc) is None:
        pytest.skip("nvcc not available")
    out = tmp_path_factory.mktemp("ptxas") / "libcheck.so"
    cmd = [nvcc, "-Xptxas=-v", *libbuild.NVCC_FLAGS, "-I" + libbuild.INCLUDE, "-I" + libbuild.CSRC,
           os.path.join(libbuild.CSRC, "moe_api.cu"), "-o", str(out)]
    res = subprocess.run(cmd, capture_output=True, text=True, check=True)
    kernels = {}
    current = None
    for line in (res.stdout + res.stderr).splitlines():
        m = ENTRY.search(line)
        if m:
            current = m.group(1)
            kernels[current] = {}
            continue
        if current is None:
            continue
        m = SPILL.search(line)
        if m:
            kernels[current]["spill"] = int(m.group(1)) + int(m.group(2))
        m = REGS.search(line)
        if m:
            kernels[current]["regs"] = int(m.group(1))
    assert kernels, "no kernels in the ptxas report"
    return kernels


def test_no_kernel_spills(ptxas_report):
    spilling = {k: v for k, v in ptxas_report.items() if v.get("spill", 0) != 0}
    assert not spilling, spilling


def test_fp8_gemm_register_split_matches_launch(ptxas_report):
    seen = set()
    for name, res in ptxas_report.items():
        m = FP8.search(name)
        if not m:
            continue
        ew = int(m.group(2))
        threads = 32 * (4 + ew)  # producer, MMA, scheduler, lender + promotion warps
        launch_regs = 65536 // threads // 8 * 8
        assert res["regs"] == launch_regs, (name, res["regs"], launch_regs)
        ctrl = 48
        epi = (launch_regs * threads - 128 * ctrl) // (32 * ew) // 8 * 8
        assert 128 * ctrl + 32 * ew * epi <= launch_regs * threads
        assert launch_regs <= epi <= 256
        seen.add((int(m.group(1)), ew, int(m.group(3))))
    # both epilogues (SwiGLU = 2, bf16 = 1) with 8 and 16 promotion warps; the
    # SwiGLU epilogue also with UE8M0 scales for h (last field 1)
    assert seen == {(1, 8, 0), (1, 16, 0), (2, 8, 0), (2, 16, 0), (2, 8, 1), (2, 16, 1)}, seen
