"""Failure detection on the GPU without a fault: a wait that nothing will
ever satisfy runs out after its time limit, the kernel reports the timeout in
its status word and returns, and the CUDA context stays usable.

Two forms: a one-CTA test kernel waiting through the product's own bounded
waiter, and the product forward kernel itself, built with FA_TEST_WITHHOLD_KV
(never in the release library), whose load warp does not load one K tile so
that the MMA thread's wait for it runs out (50 ms in that build)."""
import ctypes
import os
import subprocess

import numpy as np

import pytest
import torch

from exact_attention_forward_tiled_gb300 import api
from exact_attention_forward_tiled_gb300 import build as fa_build
from oracle import oracle as orc

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


def _fwd(L, q, k, v, o, lse, B, H, S, D):
    vp = ctypes.c_void_p
    return L.fa_fwd(vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()), vp(o.data_ptr()), vp(lse.data_ptr()),
                    B, H, S, S, D, ctypes.c_float(D ** -0.5), 0, None, None, 0, 0, api.FA_BF16, None)


def test_forward_kernel_timeout_path(cuda_device, tmp_path):
    """The forward kernel's own abort path: CTA 0 never gets K block 2 of its
    first work tile, the MMA thread's wait gives up, every role leaves (the
    load warp drains its copies, the MMA thread waits for its products, tensor
    memory is freed, the last CTA resets the scheduler counters), and the
    status word says FA_ERR_DEVICE_TIMEOUT. Afterwards, on the same context:
    64 launches of the same build (the 64th reuses the aborted launch's
    scheduler slot) and a release-build forward all match the oracle."""
    so = fa_build.build_variant(str(tmp_path / "withhold"), ["FA_TEST_WITHHOLD_KV"])
    L = ctypes.CDLL(so)
    L.fa_fwd.restype = ctypes.c_int
    L.fa_fwd.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5 + [ctypes.c_float] + [ctypes.c_int] + \
        [ctypes.c_void_p] * 2 + [ctypes.c_int] * 3 + [ctypes.c_void_p]
    L.fa_get_device_status.restype = ctypes.c_int
    L.fa_get_device_status.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]
    L.fa_test_set_withhold.argtypes = [ctypes.c_int]
    g = torch.Generator(device="cuda").manual_seed(77)
    B, H, S, D = 1, 2, 1024, 128          # 8 work tiles of 8 key blocks
    q, k, v = (torch.randn((B * S, H, D), generator=g, device="cuda").to(torch.bfloat16) for _ in range(3))
    o = torch.zeros_like(q)
    lse = torch.zeros((B, H, S), device="cuda")
    raw = ctypes.c_int(0)
    L.fa_test_set_withhold(2)
    assert _fwd(L, q, k, v, o, lse, B, H, S, D) == 0
    st = L.fa_get_device_status(None, ctypes.byref(raw))
    print(f"withheld K tile: status {st}, raw word {raw.value:#x}")
    assert st == -5 and (raw.value & 0x100), (st, hex(raw.value))
    # the same build, no tile withheld: 64 launches, each right
    L.fa_test_set_withhold(-1)
    qs, ks, vs = q[:256], k[:256], v[:256]
    ref_o, ref_l = orc.attention(qs.cpu(), ks.cpu(), vs.cpu(), scale=D ** -0.5, causal=False, nseq=1, Sq=256,
                                 Sk=256)
    o2 = torch.empty_like(qs)
    l2 = torch.empty((1, H, 256), device="cuda")
    for i in range(64):
        o2.zero_()
        assert _fwd(L, qs, ks, vs, o2, l2, 1, H, 256, D) == 0
        assert L.fa_get_device_status(None, ctypes.byref(raw)) == 0, (i, hex(raw.value))
        assert np.abs(o2.float().cpu().numpy() - ref_o).max() <= 1e-2, i
        assert np.abs(l2.cpu().numpy() - ref_l).max() <= 1e-3, i
    # and the release library on the same context
    fa_build.build()
    o3, l3 = api.attention_forward(q, k, v, batch=B)
    assert api.fa_get_device_status()[0] == 0
    ref_o, ref_l = orc.attention(q.cpu(), k.cpu(), v.cpu(), scale=D ** -0.5, causal=False, nseq=B, Sq=S, Sk=S)
    assert np.abs(o3.float().cpu().numpy() - ref_o).max() <= 1e-2
    assert np.abs(l3.cpu().numpy() - ref_l).max() <= 1e-3
