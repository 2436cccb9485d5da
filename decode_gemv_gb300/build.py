"""Build liblw.so (the C-ABI library) in-tree for sm_103a.

nvcc compiles each CUDA translation unit in parallel; g++ compiles the host
builder; nvcc links the shared library (CUDA runtime linked statically).
Output: decode_gemv_gb300/_build/liblw.so.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INC = os.path.join(ROOT, "include")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "liblw.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CU = ["lw_api.cu", "lw_q.cu", "lw_qlut.cu", "lw_bf16.cu", "lw_noalloc.cu", "lw_trans.cu",
      "lw_strips.cu"]
CPP = ["lw_host.cpp", "lw_file.cpp"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _run(cmd):
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode:
        raise RuntimeError(f"command failed: {' '.join(cmd)}\n{p.stdout}\n{p.stderr}")
    return p.stdout + p.stderr


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(OUT, exist_ok=True)
    nvcc = _nvcc()
    jobs = []
    for f in CU:
        o = os.path.join(OUT, f + ".o")
        cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
               "-I", INC, "-I", CSRC, "-c", os.path.join(CSRC, f), "-o", o]
        if ptxas_info:
            cmd.insert(1, "-Xptxas=-v")
        jobs.append((cmd, o))
    for f in CPP:
        o = os.path.join(OUT, f + ".o")
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-I", INC, "-I", CSRC,
               "-I", "/usr/local/cuda/include", "-c", os.path.join(CSRC, f), "-o", o]
        jobs.append((cmd, o))
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        logs = list(ex.map(lambda j: _run(j[0]), jobs))
    if verbose or ptxas_info:
        for (cmd, _), log in zip(jobs, logs):
            if log.strip():
                print(os.path.basename(cmd[-3]), log, file=sys.stderr)
    tmp = LIB + f".{os.getpid()}.tmp"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *[o for _, o in jobs], "-lpthread"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv))
