"""Pins of the FP8 oracle (``oracle/fp8.py``) against things other than itself.

Each ``pin_*`` takes the module (or a deliberately broken copy of it, see
``tests/test_oracle_fp8_mutants.py``) and raises AssertionError when it
disagrees with what the pages and the mathematics fix:

* the rotation is Q M with M = diag(sigma) H_D / sqrt(D), H_D from
  ``scipy.linalg.hadamard`` ("FlashAttention-3 (lukebest wiki)", technique 3,
  incoherent processing), applied to Q and K but not V;
* the block scales and codes follow their fp64 definition -- amax / 448 of
  each 128-row block after the rotation, e4m3(y / scale) -- wherever fp32
  rounding cannot decide otherwise (technique 3, block quantisation);
* where every rounding of P is exact (scores a whole number of log2 units
  apart, V block scales powers of two), the e4m3 attention equals the exact
  attention of the dequantised inputs (``oracle.attention_head``, itself
  pinned against torch's SDPA);
* a two-key case whose rounded P and output are derived by hand;
* causal rows ignore the keys they cannot see.
"""
import math

import numpy as np
import scipy.linalg

from oracle import oracle as O

U32 = 2.0 ** -24      # unit roundoff of fp32


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16_values(shape, rng, scale=1.0):
    """Random values that a bf16 tensor can hold exactly."""
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    bits = x.view(np.uint32) & np.uint32(0xFFFF0000)
    return bits.view(np.float32).astype(np.float64)


def _e4m3_boundaries():
    """Positive e4m3 values and the rounding boundaries (midpoints) between
    neighbours."""
    vals = O.E4M3_VALUES[:0x7F]
    return vals, (vals[:-1] + vals[1:]) / 2


def check_quantised(codes, scales, x, sigma, block=128):
    """Codes and scales of one (sequence, head) against the fp64 definition:
    y = x M (or x), scale_b = amax(y_b) / 448, code = e4m3(y / scale_b). fp32
    evaluation may move y / scale by at most ``err`` (the butterflies: log2 D
    roundings of sums bounded by sum |x|; the scale and multiplier: a few
    roundings), so a code may differ only where y / scale lies within ``err``
    of a rounding boundary, and then by one step."""
    x = np.asarray(x, dtype=np.float64)
    L, D = x.shape
    codes = np.asarray(codes)
    scales = np.asarray(scales, dtype=np.float64)
    nb = (L + block - 1) // block
    assert codes.shape == (L, D) and scales.shape == (nb,), (codes.shape, scales.shape)
    if sigma is not None:
        sg = np.asarray(sigma, dtype=np.float64).reshape(D)
        y = (x * sg) @ scipy.linalg.hadamard(D).astype(np.float64) / math.sqrt(D)
        stages = int(math.log2(D))
        y_err = (stages + 1) * U32 * np.abs(x).sum(axis=1, keepdims=True) / math.sqrt(D)
    else:
        y = x
        y_err = np.zeros((L, 1))
    _, mids = _e4m3_boundaries()
    for b in range(nb):
        rs = slice(b * block, min((b + 1) * block, L))
        amax = np.abs(y[rs]).max()
        if amax == 0:
            assert scales[b] == 1.0, (b, scales[b])
            assert np.all(codes[rs] & 0x7F == 0), b
            continue
        s = amax / 448.0
        s_err = 4 * U32 * s + y_err[rs].max() / 448.0
        assert abs(scales[b] - s) <= s_err, ("scale", b, scales[b], s)
        r = y[rs] / s
        err = np.abs(r) * (6 * U32 + s_err / s) + y_err[rs] / s
        ref = O.e4m3_encode(r)
        got = codes[rs]
        bad = got != ref
        if bad.any():
            a = np.abs(r[bad])
            d = np.min(np.abs(a[:, None] - mids[None, :]), axis=1)
            assert np.all(d <= err[bad]), ("code far from a boundary differs", b, int(bad.sum()))
            step = np.abs(O.e4m3_decode(got[bad]) - O.e4m3_decode(ref[bad]))
            gap = np.abs(np.diff(O.E4M3_VALUES[:0x7F])).max()
            assert np.all(step <= gap) and np.all(np.sign(O.e4m3_decode(got[bad])) * np.sign(r[bad]) >= 0), b


def pin_fwht_is_hadamard(f):
    """The butterflies compute x H_D, H_D from scipy, exactly on small
    integers in fp64 and within log2 D roundings in fp32."""
    r = _rng(0)
    for D in (1, 2, 4, 8, 16, 32, 64, 128, 256):
        x = r.integers(-50, 50, size=(5, D)).astype(np.float64)
        H = scipy.linalg.hadamard(D).astype(np.float64)
        assert np.array_equal(f.fwht(x, np.float64), x @ H), D
        x32 = _bf16_values((7, D), r)
        y32 = f.fwht(x32, np.float32).astype(np.float64)
        bound = max(1, int(math.log2(D))) * U32 * np.abs(x32).sum(axis=1, keepdims=True)
        assert np.all(np.abs(y32 - x32 @ H) <= bound), D


def pin_prepare_against_definition(f):
    """Rotation, 128-row blocks, amax after the rotation, amax / 448, e4m3:
    against the fp64 definition; ragged last block, an outlier block and an
    all-zero block included."""
    r = _rng(1)
    for D in (64, 128, 256):
        L = 300
        x = _bf16_values((L, D), r)
        x[5, 7] = 60.0                     # outlier in block 0
        x[128, 3] = -25.0                  # first row of block 1
        x[255, D - 1] = 40.0               # last row of block 1
        sigma = r.choice([-1.0, 1.0], size=D)
        for sg in (sigma, None):
            codes, scales = f.prepare(x, sg)
            check_quantised(codes, scales, x, sg)
        z = np.zeros((256, D))
        z[:128] = x[:128]
        codes, scales = f.prepare(z, sigma)
        check_quantised(codes, scales, z, sigma)


def pin_prepare_qkv_rotates_q_and_k_only(f):
    """Q and K are rotated by the same M; V keeps its own basis."""
    r = _rng(2)
    D = 128
    q, k, v = (_bf16_values((200, D), r) for _ in range(3))
    v[:, 5] *= 20.0                        # one outlier column in V
    sigma = r.choice([-1.0, 1.0], size=D)
    q8, qs, k8, ks, v8, vs = f.prepare_qkv(q, k, v, sigma)
    check_quantised(q8, qs, q, sigma)
    check_quantised(k8, ks, k, sigma)
    check_quantised(v8, vs, v, None)


def pin_dequantize_layout(f):
    """Scale b multiplies rows [128 b, 128 b + 128)."""
    codes = np.full((300, 4), 0x38, np.uint8)          # code of 1.0
    scales = np.array([0.5, 2.0, 8.0], dtype=np.float32)
    d = f.dequantize(codes, scales)
    assert np.all(d[:128] == 0.5) and np.all(d[128:256] == 2.0) and np.all(d[256:] == 8.0)


def pin_tensor_scale_and_codes(f):
    """Per-tensor comparison: scale amax / 448 of the whole tensor, codes
    e4m3(x / scale) (7.5 is the largest magnitude, so 7.5 / s = 448)."""
    x = np.array([[0.25, -7.5, 3.0], [1.0, 0.0, -2.0]])
    s = f.tensor_scale(x)
    assert s == 7.5 / 448.0
    c = f.quantize_tensor(x, s)
    assert c[0, 1] == 0xFE and c[1, 1] == 0x00
    back = O.e4m3_decode(c) * s
    assert np.all(np.abs(back - x) <= 2.0 ** -4 * np.abs(x))
    assert f.tensor_scale(np.zeros((3, 3))) == 1.0


def _exact_case(causal):
    """Codes and scales whose e4m3 P rounding is exact under the kappa = 4
    rule: every log2 score is an integer (q = e_0, k_j = n_j e_0, scale =
    ln 2) and the V block scales are powers of two. Tile 0 holds scores -4
    .. 4 (its -4 gives x = 2^-6, which an unscaled P = 2^-10 could not
    hold), tile 1 starts with a score of 10 (a move of the running max by
    more than tau = 4) and tile 2 reaches 12 (within tau: no move)."""
    r = _rng(3 + causal)
    D, L = 16, 300
    q8 = np.zeros((L, D), np.uint8)
    q8[:, 0] = O.e4m3_encode(np.array([1.0]))[0]
    n = np.concatenate([r.integers(-4, 5, 128), r.integers(6, 11, 128), r.integers(7, 13, 44)]).astype(float)
    n[0], n[1], n[128], n[256] = 4, -4, 10, 12
    k8 = np.zeros((L, D), np.uint8)
    k8[:, 0] = O.e4m3_encode(n)
    assert np.array_equal(O.e4m3_decode(k8[:, 0]), n)
    v8 = r.integers(0, 0x7E, size=(L, D)).astype(np.uint8) | (r.integers(0, 2, size=(L, D)) << 7).astype(np.uint8)
    ones = np.ones(3, np.float32)
    vs = np.array([0.5, 2.0, 0.25], np.float32)
    return q8, ones, k8, ones, v8, vs, math.log(2.0)


def pin_exact_when_rounding_is_exact(f):
    """Where every e4m3 rounding of P is exact, the FP8 attention equals the
    exact attention of the dequantised inputs (lazy rescale, kappa, the V
    weights and the final division are then all exact)."""
    for causal in (False, True):
        q8, qs, k8, ks, v8, vs, scale = _exact_case(causal)
        L = q8.shape[0]
        rows = np.arange(L)
        o, lse = f.attention_fp8(q8, qs, k8, ks, v8, vs, rows, L, scale=scale, causal=causal)
        qd, kd, vd = f.dequantize(q8, qs), f.dequantize(k8, ks), f.dequantize(v8, vs)
        o_ref, lse_ref = O.attention_head(qd, rows, kd, vd, L, scale, causal)
        assert np.abs(o - o_ref).max() <= 1e-12 * np.abs(vd).max(), causal
        assert np.abs(lse - lse_ref).max() <= 1e-12, causal


def pin_two_keys_by_hand(f):
    """One query, two keys with P = 1 and P = 1.2 * 2^-8 against the row max.
    Scaled by 2^4 the second is 1.2 * 2^-4, whose nearest e4m3 neighbours are
    1.125 * 2^-4 and 1.25 * 2^-4: it rounds to 1.25 * 2^-4. So
    O = (v0 + 1.25 * 2^-8 v1) / (1 + 1.2 * 2^-8), l summing the unrounded P,
    and LSE = ln(1 + 1.2 * 2^-8)."""
    D = 8
    one = O.e4m3_encode(np.array([1.0]))[0]
    m_one = O.e4m3_encode(np.array([-1.0]))[0]
    q8 = np.zeros((1, D), np.uint8)
    q8[0, 0] = one
    k8 = np.zeros((2, D), np.uint8)
    k8[1, 0] = m_one
    t1 = math.log2(1.2) - 8.0                 # log2 of the second P
    scale = -t1 * math.log(2.0)               # the second score, -scale, is t1 in log2 units
    v8 = O.e4m3_encode(np.array([[1.0, -2.0, 0.5, 3.0, -0.25, 6.0, 1.5, -4.0],
                                 [-3.0, 4.0, 2.0, -1.0, 8.0, -0.5, 0.75, 1.0]]))
    vs = np.array([0.25], np.float32)
    sc = np.ones(1, np.float32)
    o, lse = f.attention_fp8(q8, sc, k8, sc, v8, vs, np.array([0]), 1, scale=scale, causal=False)
    v = O.e4m3_decode(v8) * 0.25
    ref = (v[0] + 1.25 * 2.0 ** -8 * v[1]) / (1.0 + 1.2 * 2.0 ** -8)
    assert np.abs(o[0] - ref).max() <= 1e-14, (o[0], ref)
    assert abs(lse[0] - math.log(1.0 + 1.2 * 2.0 ** -8)) <= 1e-14


def pin_causal_rows_ignore_invisible_keys(f):
    """Row i of a causal problem with Lq < Lk sees keys j <= i + Lk - Lq:
    changing the keys and values it cannot see leaves it bit-identical, and
    changing the last key it can see does not."""
    r = _rng(5)
    D, Lq, Lk = 64, 150, 300
    q, k, v = (_bf16_values((n, D), r) for n in (Lq, Lk, Lk))
    sigma = r.choice([-1.0, 1.0], size=D)
    q8, qs, k8, ks, v8, vs = f.prepare_qkv(q, k, v, sigma)
    rows = np.array([0, 77, 149])
    o, lse = f.attention_fp8(q8, qs, k8, ks, v8, vs, rows, Lq, scale=0.125, causal=True)
    for n, i in enumerate(rows):
        last = i + Lk - Lq
        k2, v2 = k8.copy(), v8.copy()
        k2[last + 1:] = 0x40
        v2[last + 1:] = 0xC0
        # the same rows in every call: BLAS may round a product of another
        # shape differently
        o2, lse2 = f.attention_fp8(q8, qs, k2, ks, v2, vs, rows, Lq, scale=0.125, causal=True)
        assert np.array_equal(o2[n], o[n]) and lse2[n] == lse[n], i
        k3 = k8.copy()
        k3[last] ^= 0x08
        o3, _ = f.attention_fp8(q8, qs, k3, ks, v8, vs, rows, Lq, scale=0.125, causal=True)
        assert not np.array_equal(o3[n], o[n]), i


ALL_PINS = [pin_fwht_is_hadamard, pin_prepare_against_definition, pin_prepare_qkv_rotates_q_and_k_only,
            pin_dequantize_layout, pin_tensor_scale_and_codes, pin_exact_when_rounding_is_exact,
            pin_two_keys_by_hand, pin_causal_rows_ignore_invisible_keys]
