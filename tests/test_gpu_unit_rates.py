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


def test_tma_small_box_issue(cuda_device, tmp_path):
    """Small TMA boxes (16 rows x 128 bytes, the paged K/V box at 16-key pages)
    from one warp against several warps with the same bytes in flight. Prints
    GB/s per configuration; asserts only that every run finished."""
    so = str(tmp_path / "tma_issue.so")
    subprocess.run([fa_build.nvcc(), *fa_build.ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                    "-cudart", "shared", os.path.join(HERE, "gpu_helpers", "tma_issue.cu"), "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.tma_issue_rate.restype = ctypes.c_double
    lib.tma_issue_rate.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 6 + [ctypes.c_void_p]
    rows = 262144                                  # [rows, 2048] bf16 = 1 GiB, rows of 4 KB
    buf = torch.zeros(rows * 2048, dtype=torch.bfloat16, device=cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for box_rows, warps, ops in [(16, 1, 16), (16, 1, 32), (16, 2, 16), (16, 4, 8), (64, 1, 8), (128, 1, 4)]:
        per_batch = sms * warps * ops * box_rows * 128
        batches = max(4, (4 << 30) // per_batch)
        gbs = lib.tma_issue_rate(buf.data_ptr(), rows, box_rows, warps, ops, batches, sms, err.data_ptr())
        torch.cuda.synchronize()
        print(f"box {box_rows:3d} rows x 128 B, {warps} warp(s) x {ops:2d} boxes in flight "
              f"({warps * ops * box_rows * 128 // 1024:3d} KB per SM): {gbs:8.1f} GB/s")
        assert gbs > 0.0, gbs
    assert int(err.item()) == 0


def test_mma_issue_rate(cuda_device, tmp_path):
    """Back-to-back tcgen05.mma M128 N128 K16 (bf16) from one thread per SM,
    descriptors built as in the forward kernel: cycles per product for the
    QK^T form (both operands in shared memory) and the PV form (A in tensor
    memory, B MN-major). Nominal: 64 cycles (8192 dense bf16 FLOP per clock
    per SM). Prints; asserts only that the runs finished."""
    so = str(tmp_path / "mma_issue.so")
    csrc = os.path.join(os.path.dirname(HERE), "exact_attention_forward_tiled_gb300", "csrc")
    subprocess.run([fa_build.nvcc(), *fa_build.ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                    "-cudart", "shared", "-I", csrc, os.path.join(HERE, "gpu_helpers", "mma_issue.cu"), "-o", so],
                   check=True)
    lib = ctypes.CDLL(so)
    lib.mma_issue_cycles.restype = ctypes.c_double
    lib.mma_issue_cycles.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cyc = torch.zeros(sms, dtype=torch.int64, device=cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    for form, name in ((0, "QK^T form (SS, B K-major)"), (1, "PV form (A in tensor memory, B MN-major)")):
        lib.mma_issue_cycles(form, 16, sms, cyc.data_ptr(), err.data_ptr())
        c = lib.mma_issue_cycles(form, 2048, sms, cyc.data_ptr(), err.data_ptr())
        print(f"{name:42s} {c:6.1f} cycles per M128 N128 K16 product ({64.0 / c * 100:5.1f} % of nominal)")
        assert c > 0.0, c
    assert int(err.item()) == 0


def test_fp8_prep_rates(cuda_device):
    """fa_fp8_prep throughput at D = 64 / 128 / 256 with the same bytes (bf16
    Q, K, V of 4 x 8192 tokens, H = 32 / 16 / 8): GB/s of the algorithmic
    bytes (3 per element: 2 read, 1 written), CUDA events around 50 calls.
    Prints; asserts only that the calls ran."""
    from exact_attention_forward_tiled_gb300 import api
    from exact_attention_forward_tiled_gb300 import build as fa_build_mod
    fa_build_mod.build()
    g = torch.Generator(device=cuda_device).manual_seed(0)
    for H, D in ((32, 64), (16, 128), (8, 256)):
        B, S = 4, 8192
        q, k, v = (torch.randn((B * S, H, D), generator=g, device=cuda_device).to(torch.bfloat16) for _ in range(3))
        sigma = (torch.randint(0, 2, (D,), generator=g, device=cuda_device, dtype=torch.int32) * 2 - 1).to(torch.int8)
        prep = api.fp8_prepare(q, k, v, sigma, batch=B)

        def run():
            api.fa_fp8_prep(q, k, v, prep["q8"], prep["k8"], prep["v8"], prep["q_scale"], prep["k_scale"],
                            prep["v_scale"], sigma, B, H, S, S, D)
        for _ in range(5):
            run()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(50):
            run()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / 50
        gbs = 3 * 3 * B * S * H * D / (ms * 1e-3) / 1e9
        print(f"fa_fp8_prep D = {D:3d}: {ms * 1e3:7.1f} us per call, {gbs:7.0f} GB/s")
        api.fa_get_device_status()
        assert gbs > 0.0
