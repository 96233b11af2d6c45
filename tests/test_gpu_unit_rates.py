"""Measurement (no parity): per-SM issue rates of MUFU ex2 and the FMA pipe on
this GPU, so the exponential-versus-matmul budget (the FlashAttention-3 essay's
MUFU paragraph, 3.9 vs 989 TFLOP/s on H100) is a number here, not an
assumption. Prints the rates; asserts only that they are sane."""
import ctypes
import os
import subprocess

import pytest
import torch

from exact_attention_forward_tiled_gb300 import build as fa_build

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_unit_rates(cuda_device, tmp_path):
    so = str(tmp_path / "unit_rates.so")
    subprocess.run([fa_build.nvcc(), *fa_build.ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                    "-cudart", "shared", os.path.join(HERE, "gpu_helpers", "unit_rates.cu"), "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.unit_rate.restype = ctypes.c_double
    lib.unit_rate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    names = ["ex2.approx.f32 (MUFU)", "ex2.approx.f16x2 (MUFU, 2 results)", "fma.rn.f32", "fma.rn.f32x2 (2 results)"]
    rates = {}
    for kind, name in enumerate(names):
        lib.unit_rate(kind, sms, 64)                    # warm-up
        rates[name] = lib.unit_rate(kind, sms, 4096)
        print(f"{name:40s} {rates[name]:8.2f} instructions / clock / SM")
    for r in rates.values():
        assert 1.0 <= r <= 1024.0
