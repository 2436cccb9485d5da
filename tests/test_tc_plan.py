"""The tensor-core products' work split (decode_gemv_gb300/csrc/lw_tcplan.h),
on the CPU: tests/tc_plan_check.cpp is built against the library's own header
with the plain C++ compiler and checks the contiguous per-CTA ranges, the
owners of every row block and the grid choice over a sweep of launch shapes
(see its header).  No GPU."""
import shutil
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent


def test_tc_plan(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = tmp_path / "tc_plan_check"
    subprocess.run([cxx, "-std=c++17", "-O2", "-Wall", "-Wextra", "-Werror",
                    "-I", str(ROOT / "decode_gemv_gb300" / "csrc"),
                    str(ROOT / "tests" / "tc_plan_check.cpp"), "-o", str(exe)],
                   check=True, capture_output=True, text=True, timeout=300)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok "), r.stdout
