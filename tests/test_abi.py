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
    for code in range(0, -10, -1):
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
    # no key rows at all: k and v may be NULL (the host checks pass)
    assert _call(L, k=None, v=None, Sk=0) == -7
    assert _call(L, k=None, Sk=128) == -1
    raw = ctypes.c_int(0)
    assert L.fa_get_device_status(None, ctypes.byref(raw)) == -7


def _fp8_varlen(L, cq=0x6000, ck=0x7000, cbq=0x8000, cbk=0x9000, tq=300, tk=300, mq=128, mk=128, D=128,
                o=0x4000, scale=0.1):
    return L.fa_fwd_fp8_varlen(0x1000, 0x2000, 0x3000, 0xa000, 0xb000, 0xc000, o, 0x5000, 2, 2, cq, ck, cbq,
                               cbk, tq, tk, mq, mk, D, ctypes.c_float(scale), 0, None)


def _prep_varlen(L, q=0x1000, k=0x2000, cq=0x6000, ck=0x7000, cbq=0x8000, cbk=0x9000, mq=128, mk=128, D=128,
                 dtype=api.FA_BF16, qs=0xa000):
    return L.fa_fp8_prep_varlen(q, k, 0x3000, dtype, 0x11000, 0x12000, 0x13000, qs, 0xb000, 0xc000, None, 2, 2,
                                cq, ck, cbq, cbk, 300, 300, mq, mk, D, None)


def test_fp8_varlen_host_argument_checks(L):
    # every cu_seqlens / cu_blocks array is required by the forward
    for kw in ("cq", "ck", "cbq", "cbk"):
        assert _fp8_varlen(L, **{kw: None}) == -1, kw
    assert _fp8_varlen(L, D=96) == -2                # head sizes 64, 128, 256 only
    assert _fp8_varlen(L, tq=-1) == -1 and _fp8_varlen(L, scale=-2.0) == -1
    assert _fp8_varlen(L, o=0x4008) == -3
    assert _fp8_varlen(L, mq=0) == 0                   # no query rows: a no-op
    # the preparation needs the arrays of each side it prepares, and only those
    assert _prep_varlen(L, cq=None) == -1 and _prep_varlen(L, cbk=None) == -1
    assert _prep_varlen(L, dtype=api.FA_FP8_E4M3) == -2 and _prep_varlen(L, D=96) == -2
    assert _prep_varlen(L, q=0x1004) == -3 and _prep_varlen(L, qs=0xa002) == -3
    assert _prep_varlen(L, mq=0, mk=0) == 0
    assert L.fa_varlen_blocks(None, 3, 0x8000, None) == -1 and L.fa_varlen_blocks(0x6000, -1, 0x8000, None) == -1
    import torch
    if not torch.cuda.is_available():
        assert _fp8_varlen(L) == -7 and _prep_varlen(L) == -7 and _prep_varlen(L, q=None, cq=None, mq=0) == -7
