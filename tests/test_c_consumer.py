"""include/lw.h is plain C and liblw.so serves a C caller with no Python or
PyTorch in the process: tests/c_consumer.c is compiled as strict C11
against the header, linked against the library and run on the CPU (host
entry points only: encode, sections, validation, bundle strings)."""
import os
import shutil
import subprocess

import pytest

from decode_gemv_gb300 import lw

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def built():
    if not os.path.exists(lw.LIB_PATH):
        from decode_gemv_gb300 import build
        build.build()
    return lw.LIB_PATH


def test_plain_c_caller(built, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "c_consumer"
    libdir = os.path.dirname(built)
    subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_consumer.c"),
                    "-L", libdir, "-llw", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
