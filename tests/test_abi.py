"""CPU tests of the C-ABI library: it builds, loads, exports every function the
header declares, and rejects bad arguments on the host without touching a GPU."""
import ctypes
import subprocess

import pytest

from exact_attention_forward_tiled_gb300 import api
from exact_attention_forward_tiled_gb300 import build as fa_build


@pytest.fixture(scope="module")
def L():
    fa_build.build()
    return api.lib()


def test_header_symbols_exported(L):
    names = api.header_functions()
    assert {"fa_fwd", "fa_get_device_status", "fa_strerror", "fa_version"} <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", api.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for n in names:
        assert n in exported, n
        assert hasattr(L, n)


def test_version_and_strerror(L):
    assert api.fa_version() >> 16 == 1
    for code in range(0, -8, -1):
        assert api.strerror(code) not in ("", "unknown status")
    assert api.strerror(-99) == "unknown status"


def _call(L, q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=1, H=2, Sq=128, Sk=128, D=128,
          scale=0.1, causal=0, cq=None, ck=None, tq=0, tk=0, dtype=api.FA_BF16):
    # fake, never-dereferenced device addresses: only host-side checks run
    return L.fa_fwd(q, k, v, o, lse, B, H, Sq, Sk, D, ctypes.c_float(scale), causal, cq, ck, tq, tk,
                    dtype, None)


def test_host_argument_checks(L):
    assert _call(L, D=96) == -2 and _call(L, D=32) == -2
    assert _call(L, dtype=api.FA_FP8_E4M3) == -2
    assert _call(L, dtype=7) == -1
    assert _call(L, H=0) == -1 and _call(L, B=-1) == -1 and _call(L, Sq=-3) == -1
    assert _call(L, scale=float("nan")) == -1 and _call(L, scale=-1.0) == -1
    assert _call(L, causal=2) == -1
    assert _call(L, cq=0x6000) == -1                 # one of the two cu_seqlens
    assert _call(L, cq=0x6000, ck=0x7000, tq=-1) == -1
    assert _call(L, q=0x1008) == -3 and _call(L, o=0x4004) == -3 and _call(L, lse=0x5002) == -3
    assert _call(L, q=None) == -1 and _call(L, lse=None) == -1
    assert _call(L, B=70000, Sq=70000) == -1        # more than 2^31 tokens
    # empty problems are a successful no-op
    assert _call(L, B=0) == 0 and _call(L, Sq=0) == 0


def test_valid_call_without_gpu_reports_no_device(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _call(L) == -7
    raw = ctypes.c_int(0)
    assert L.fa_get_device_status(None, ctypes.byref(raw)) == -7
