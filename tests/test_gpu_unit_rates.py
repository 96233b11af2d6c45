"""Per-SM issue rates of MUFU ex2 and the FMA pipe on this GPU, so the
exponential-versus-matmul budget (the FlashAttention-3 essay's MUFU
paragraph, 3.9 vs 989 TFLOP/s on H100) is a number here, not an assumption.

Expected, and asserted: an SM has 128 fp32 lanes (4 sub-partitions x 32), so
fma.rn.f32 issues at most 128 results per clock and fma.rn.f32x2 at most 64
instructions (128 results); MUFU delivers 32 ex2.approx.f32 results per clock
per SM on GB300 (8 per sub-partition), the same 32 results when they come as
ex2.approx.f16x2 pairs (16 instructions). A rate more than 15 % below these
means the measurement, or the unit, is not what the softmax budget assumes."""
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
    expect = dict(zip(names, (32.0, 16.0, 128.0, 64.0)))
    for name, r in rates.items():
        assert 0.85 * expect[name] <= r <= 1.02 * expect[name], (name, r, expect[name])
