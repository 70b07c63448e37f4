"""The C ABI from plain C: tests/c/abi_from_c.c compiles as C99 against
include/dspark.h with warnings as errors, links against libdspark.so and runs
host-side checks only (no kernel launch), so it needs no GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INC = "/usr/local/cuda/include"


def test_header_and_library_work_from_c(tmp_path):
    from serving_draft_verify_gb300 import build as b
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    if not os.path.exists(b.LIB):
        b.build()
    lib = b.LIB
    exe = tmp_path / "abi_from_c"
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "abi_from_c.c"), "-o", str(exe),
           "-L", os.path.dirname(lib), "-ldspark", "-Wl,-rpath," + os.path.dirname(lib)]
    if os.path.isdir(CUDA_INC):
        cmd[5:5] = ["-I", CUDA_INC]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
