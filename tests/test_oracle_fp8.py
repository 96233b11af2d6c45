"""CPU tests of the oracle's Hadamard rotation, E4M3 codec and FP8 path
(``oracle/fp8.py``): every pin of ``tests/fp8_pins.py`` on the real module."""
import numpy as np
import pytest
import scipy.linalg
import torch

from oracle import fp8 as F
from oracle import oracle as O
from tests.fp8_pins import ALL_PINS


@pytest.mark.parametrize("D", [1, 2, 4, 8, 16, 32, 64, 128, 256])
def test_hadamard_matches_scipy(D):
    h = O.hadamard(D)
    assert np.array_equal(h, scipy.linalg.hadamard(D).astype(np.float64))
    assert np.array_equal(h @ h.T, D * np.eye(D))


@pytest.mark.parametrize("D", [64, 128, 256])
def test_rotation_is_orthogonal_and_preserves_scores(D):
    """(QM)(KM)^T = QK^T for M = Hadamard x random signs (wiki, section 3)."""
    r = np.random.default_rng(D)
    sigma = r.choice([-1.0, 1.0], size=D)
    M = O.rotation(sigma)
    assert np.abs(M @ M.T - np.eye(D)).max() < 1e-14
    q, k, v = r.standard_normal((33, D)), r.standard_normal((47, D)), r.standard_normal((47, D))
    assert np.abs((q @ M) @ (k @ M).T - q @ k.T).max() < 1e-12
    a = O.attention_head(q, np.arange(33), k, v, 33, D ** -0.5, False)
    b = O.attention_head(q @ M, np.arange(33), k @ M, v, 33, D ** -0.5, False)
    assert np.abs(a[0] - b[0]).max() < 1e-12


def test_rotation_rejects_non_power_of_two():
    with pytest.raises(ValueError):
        O.hadamard(96)


def _torch_codes(x):
    t = torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_e4m3_decode_exhaustive():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = O.e4m3_decode(np.arange(256))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9 and mine[0x08] == 2.0 ** -6


def test_e4m3_encode_values_midpoints_and_random():
    vals = O.E4M3_VALUES[:0x7F]
    mids = (vals[:-1] + vals[1:]) / 2            # ties: exact in fp32
    r = np.random.default_rng(0)
    rnd = r.uniform(-448, 448, size=20000) * r.choice([1, 1e-1, 1e-2, 1e-3], size=20000)
    for x in (vals, -vals[1:], mids, -mids, rnd):
        x32 = np.asarray(x, dtype=np.float32).astype(np.float64)
        assert np.array_equal(O.e4m3_encode(x32), _torch_codes(x32)), "encode disagrees with torch"


def test_e4m3_saturates_and_nan():
    assert O.e4m3_encode(np.array([449.0, 1e9, 464.0]))[0] == 0x7E
    assert np.all(O.e4m3_encode(np.array([449.0, 1e9, 464.0])) == 0x7E)
    assert np.all(O.e4m3_encode(np.array([-449.0, -1e9])) == 0xFE)
    assert O.e4m3_encode(np.array([np.nan]))[0] == 0x7F


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_fp8_oracle_pin(pin):
    pin(F)


def test_fp8_prepare_decides_codes_in_fp32():
    """The codes are the e4m3 rounding of fp32(y * multiplier): the same
    values from torch's float8_e4m3fn cast of the fp32 products."""
    r = np.random.default_rng(9)
    D = 128
    x = (r.standard_normal((256, D)) * 3).astype(np.float32)
    x = (x.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)
    sigma = r.choice([-1.0, 1.0], size=D)
    codes, scales = F.prepare(x, sigma)
    y = F.fwht((x * sigma).astype(np.float32), np.float32)
    norm = F.rotation_norm(D)
    for b in range(2):
        mult = norm / scales[b]
        prod = (y[b * 128:(b + 1) * 128] * mult).astype(np.float32)
        assert np.array_equal(codes[b * 128:(b + 1) * 128], _torch_codes(prod))
