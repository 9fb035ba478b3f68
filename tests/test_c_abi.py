"""The C ABI used from C alone: tests/c_abi/na3d_c_check.c includes
include/na3d.h, links libna3d.so and the CUDA runtime, and checks closed-form
results and status codes (see its header). The CPU test compiles and links it;
the GPU test runs it."""
import os
import shutil
import subprocess

import pytest

import neighborhood_attention_video_gb300 as na
from neighborhood_attention_video_gb300 import build as na_build

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "c_abi", "na3d_c_check.c")
OUT_DIR = os.path.join(HERE, "c_abi", "_build")
EXE = os.path.join(OUT_DIR, "na3d_c_check")


def build_c_check() -> str:
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    lib = na_build.build()
    os.makedirs(OUT_DIR, exist_ok=True)
    libdir = os.path.dirname(lib)
    cmd = [nvcc, "-O2", "-I", na_build.INCLUDE, SRC, "-o", EXE, "-L", libdir, "-lna3d",
           "-Xlinker", "-rpath," + libdir, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stdout + res.stderr
    return EXE


def test_c_program_compiles_and_links():
    assert os.access(build_c_check(), os.X_OK)


@pytest.mark.gpu
def test_c_program_runs_its_checks():
    exe = build_c_check()
    res = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    print(res.stdout)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "all checks passed" in res.stdout
    assert na.library_path() and os.path.exists(na.library_path())
