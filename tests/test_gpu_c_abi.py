"""The C ABI from C++ alone: tests/c/abi_smoke.cpp includes only the CUDA
runtime and include/ddp_ring.h, links libddp_ring.so, and checks the fused,
literal and tree-shaped all-reduce, a reduce-scatter, a Reducer and the error
calls on exact small-integer data (no Python, no torch in that process)."""
import os
import subprocess

import pytest

from ring_all_reduce_ddp_gb300 import build as B

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_drives_the_library(tmp_path):
    lib = B.build_library()
    exe = tmp_path / "abi_smoke"
    cmd = [B.nvcc(), *B.ARCH, "-O2", "-std=c++17", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "abi_smoke.cpp"), "-L", os.path.dirname(lib), "-lddp_ring",
           "-Xlinker", "-rpath", "-Xlinker", os.path.dirname(lib), "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]
