"""Host check of the work-tile order shared by the forward and backward
kernels (fa::tile_order in csrc/fa_internal.h): a bijection from tile indices
to (head, rank) pairs for every group size, heads visited group by group and
ranks in order within a group. Compiled with the host compiler; no GPU."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "exact_attention_forward_tiled_gb300", "csrc")


def _cuda_include():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    inc = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "include")
    return inc if os.path.exists(os.path.join(inc, "cuda_runtime.h")) else None


def test_tile_order_is_a_grouped_bijection(tmp_path):
    inc = _cuda_include()
    if inc is None or shutil.which("g++") is None:
        pytest.skip("needs g++ and the CUDA headers")
    exe = str(tmp_path / "tile_order_check")
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", CSRC, "-I", inc,
                    os.path.join(HERE, "host_helpers", "tile_order_check.cpp"), "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout
