"""Plant plausible mistakes in the oracle's C source (on the CPU, in a temporary
copy) and check that the pins catch every one of them."""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest

from tests.oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "attention_oracle.c")

MUTANTS = {
    "causal_top_left": ("int64_t lim = i + Lk - Lq + 1;", "int64_t lim = i + 1;"),
    "causal_off_by_one": ("int64_t lim = i + Lk - Lq + 1;", "int64_t lim = i + Lk - Lq;"),
    "scale_dropped": ("s[j] = scale * acc;", "s[j] = acc;"),
    "lse_without_max": ("lse[r] = m + log(l);", "lse[r] = log(l);"),
    "not_normalised": ("orow[d] /= l;", "orow[d] /= 1.0;"),
    "exp_sign_flipped": ("s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    "no_max_subtraction": ("s[j] = exp(s[j] - m);", "s[j] = exp(s[j]);"),
    "k_row_stride": ("const double *kj = k + (size_t)j * D;", "const double *kj = k + (size_t)j;"),
    "v_rows_reversed": ("const double *vj = v + (size_t)j * D;",
                        "const double *vj = v + (size_t)(visible - 1 - j) * D;"),
    "empty_row_not_zero": ("for (int d = 0; d < D; ++d) orow[d] = 0.0;\n                lse[r] = -INFINITY;",
                           "for (int d = 0; d < D; ++d) orow[d] = 1.0;\n                lse[r] = 0.0;"),
}


def _build_mutant(name, tmp):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    path_c = os.path.join(tmp, f"{name}.c")
    path_so = os.path.join(tmp, f"{name}.so")
    with open(path_c, "w") as f:
        f.write(src.replace(old, new, 1))
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", path_c, "-o", path_so, "-lm"],
                   check=True)
    lib = ctypes.CDLL(path_so)
    fn = lib.oracle_attention_rows
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                   ctypes.c_void_p, ctypes.c_void_p]

    def att(q, qpos, k, v, Lq, scale, causal):
        q = np.ascontiguousarray(q, dtype=np.float64)
        k = np.ascontiguousarray(k, dtype=np.float64)
        v = np.ascontiguousarray(v, dtype=np.float64)
        qpos = np.ascontiguousarray(qpos, dtype=np.int64)
        o = np.empty_like(q)
        lse = np.empty(q.shape[0])
        fn(q.ctypes.data, qpos.ctypes.data, q.shape[0], k.ctypes.data, v.ctypes.data, k.shape[0],
           int(Lq), q.shape[1], float(scale), int(bool(causal)), o.ctypes.data, lse.ctypes.data)
        return o, lse

    return att


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    with tempfile.TemporaryDirectory() as tmp:
        att = _build_mutant(name, tmp)
        caught = []
        for pin in ALL_PINS:
            try:
                with np.errstate(all="ignore"):
                    pin(att)
            except (AssertionError, FloatingPointError, ValueError):
                caught.append(pin.__name__)
        assert caught, f"no pin catches mutant {name}"


def test_unmutated_copy_passes_every_pin():
    """The harness itself: the unchanged source, built the same way, passes."""
    MUTANTS["_identity"] = ("return status;", "return status;")
    try:
        with tempfile.TemporaryDirectory() as tmp:
            att = _build_mutant("_identity", tmp)
            for pin in ALL_PINS:
                pin(att)
    finally:
        del MUTANTS["_identity"]
