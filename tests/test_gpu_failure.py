"""Failure detection on the GPU without a fault: a wait that nothing will
ever satisfy runs out after its time limit, the kernel reports the timeout in
its status word and returns, and the CUDA context stays usable."""
import ctypes
import os
import subprocess

import pytest
import torch

from exact_attention_forward_tiled_gb300 import api
from exact_attention_forward_tiled_gb300 import build as fa_build

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_bounded_wait_times_out_and_reports(cuda_device, tmp_path):
    src = os.path.join(HERE, "gpu_helpers", "wait_timeout.cu")
    so = str(tmp_path / "wait_timeout.so")
    subprocess.run([fa_build.nvcc(), *fa_build.ARCH, "-O2", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                    "-cudart", "shared", "-I", fa_build.CSRC, "-I", fa_build.INCLUDE, src, "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.run_wait_on_nothing.restype = ctypes.c_int
    lib.run_wait_on_nothing.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    result = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    rc = lib.run_wait_on_nothing(ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(result.data_ptr()))
    assert rc == 0                                   # no CUDA error: the kernel returned
    assert result.tolist() == [0, 1]                 # the wait gave up and raised the abort flag
    assert status.item() == 0x100 | 11               # timeout code | where it waited
    # the context is still usable: an attention forward runs and is right
    fa_build.build()
    q = torch.randn((256, 2, 64), device="cuda").to(torch.float16)
    o, lse = api.attention_forward(q, q, q, batch=1)
    assert api.fa_get_device_status()[0] == 0
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.float().transpose(0, 1)[None], q.float().transpose(0, 1)[None], q.float().transpose(0, 1)[None])
    assert (o.float().transpose(0, 1)[None] - ref).abs().max().item() <= 2e-3
