"""The grouped GEMMs' tile walk (decode_tile, csrc/moe_tile.cuh) compiled for
the host and run over random group sizes, in the plain and the interleaved
order: every (group, row tile, column tile) is named by exactly one linear
index, the streamed flag marks exactly the single-tile groups' tiles, and the
dense : sparse ratio holds in every window of 152 consecutive indices
(tests/native/tile_order_check.cpp)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "mixture_experts_ffn_route_gb300", "csrc")
SRC = os.path.join(ROOT, "tests", "native", "tile_order_check.cpp")


def _cuda_include():
    for base in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if base and os.path.exists(os.path.join(base, "include", "cuda_runtime.h")):
            return os.path.join(base, "include")
    nvcc = shutil.which("nvcc")
    if nvcc:
        inc = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "include")
        if os.path.exists(os.path.join(inc, "cuda_runtime.h")):
            return inc
    return None


def test_tile_walk_names_every_tile_once(tmp_path):
    cxx = shutil.which("g++")
    inc = _cuda_include()
    if cxx is None or inc is None:
        pytest.skip("needs g++ and the CUDA headers")
    exe = str(tmp_path / "tile_order_check")
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, "-I", inc, SRC, "-o", exe], check=True,
                   capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 failures" in r.stdout
