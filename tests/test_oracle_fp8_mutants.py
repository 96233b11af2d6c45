"""Plant plausible mistakes in a copy of the FP8 oracle (``oracle/fp8.py``, on
the CPU, in a temporary module) and check that the pins of
``tests/fp8_pins.py`` catch every one of them."""
import importlib.util
import os
import tempfile

import numpy as np
import pytest

from tests.fp8_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "fp8.py")

MUTANTS = {
    # V rotated like Q and K
    "v_rotated": ("v8, vs = prepare(v, None, block)", "v8, vs = prepare(v, sigma, block)"),
    # the block scale taken from the input before the rotation
    "scale_before_rotation": ("amax = F32(np.abs(y[rows]).max()) * norm", "amax = F32(np.abs(x32[rows]).max())"),
    # kappa dropped: P rounded without its 2^kappa headroom
    "kappa_dropped": ("x = p * (2.0 ** kappa * vs[j] / v_ref)", "x = p * (vs[j] / v_ref)\n        kappa = 0.0"),
    # block boundaries shifted by one row
    "block_shift": ("rows = slice(b * block, min((b + 1) * block, L))",
                    "rows = slice(b * block + (1 if b else 0), min((b + 1) * block + 1, L))"),
    "dequant_block_shift": ("sc = np.repeat(np.asarray(scales, dtype=np.float64), block)[:val.shape[0]]",
                            "sc = np.repeat(np.asarray(scales, dtype=np.float64), block)[1:val.shape[0] + 1]"),
    # the V block weight left out of P
    "v_weight_dropped": ("x = p * (2.0 ** kappa * vs[j] / v_ref)", "x = p * (2.0 ** kappa)"),
    # the accumulated O not rescaled when the running max moves
    "acc_not_rescaled": ("acc *= f[:, None]\n", "\n"),
    # l summed from the rounded P
    "l_from_rounded_p": ("l += p.sum(axis=1)", "l += (p8 / (2.0 ** kappa * vs[j] / v_ref)).sum(axis=1)"),
    # signs applied after the Hadamard transform (M = H diag(sigma))
    "signs_after_hadamard": ("y = fwht(x32 * sg, F32)", "y = fwht(x32, F32) * sg"),
    # 1/sqrt(D) left out of the rotation
    "norm_dropped": ("norm = rotation_norm(D)", "norm = F32(1.0)"),
    # causal mask aligned top-left instead of bottom-right
    "causal_top_left": ("np.minimum(Lk, rows + Lk - Lq + 1)", "np.minimum(Lk, rows + 1)"),
    # a butterfly with the wrong sign
    "butterfly_sign": ("y[..., 1, :] = a - b", "y[..., 1, :] = b - a"),
}


def _load_mutant(name, tmp):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    src = src.replace(old, new, 1).replace("from .oracle import", "from oracle.oracle import")
    path = os.path.join(tmp, f"fp8_{name}.py")
    with open(path, "w") as f:
        f.write(src)
    spec = importlib.util.spec_from_file_location(f"fp8_mutant_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_fp8_pins_catch_mutant(name):
    with tempfile.TemporaryDirectory() as tmp:
        mod = _load_mutant(name, tmp)
        caught = []
        for pin in ALL_PINS:
            try:
                with np.errstate(all="ignore"):
                    pin(mod)
            except (AssertionError, FloatingPointError, ValueError, IndexError):
                caught.append(pin.__name__)
        assert caught, f"no pin catches mutant {name}"


def test_unmutated_copy_passes_every_pin():
    """The harness itself: the unchanged source, loaded the same way, passes."""
    MUTANTS["_identity"] = ("TAU = 4.0", "TAU = 4.0")
    try:
        with tempfile.TemporaryDirectory() as tmp:
            mod = _load_mutant("_identity", tmp)
            for pin in ALL_PINS:
                pin(mod)
    finally:
        del MUTANTS["_identity"]
