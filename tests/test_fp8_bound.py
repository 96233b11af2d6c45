"""CPU tests of the element-wise FP8 error bounds (``tests/fp8_bound.py``)
that the GPU FP8 parity tests use."""
import numpy as np
import pytest

from oracle import fp8 as F
from oracle import oracle as O
from tests import fp8_bound as B


def test_rel_err_bounds_every_rounding():
    """|e4m3(x) - x| <= r(x) x for x over the whole range below 448, and the
    bound is tight: a midpoint just above a power of two comes within 6 % of
    2^-4, and a value just under 2^-10 loses all of itself."""
    r = np.random.default_rng(0)
    x = np.exp2(r.uniform(-14, np.log2(440.0), size=200000))
    err = np.abs(O.e4m3_round(x) - x)
    assert np.all(err <= B.e4m3_rel_err(x) * x * (1 + 1e-12))
    mid = 1.0625                                        # between 1 and 1.125
    assert abs(O.e4m3_round(np.array([mid]))[0] - mid) / mid == 2.0 ** -4 / mid
    assert B.e4m3_rel_err(np.array([mid]))[0] == 2.0 ** -4
    tiny = 2.0 ** -10 * 0.999
    assert O.e4m3_round(np.array([tiny]))[0] == 0.0 and B.e4m3_rel_err(np.array([tiny]))[0] == 1.0


def test_near_boundary_against_brute_force():
    r = np.random.default_rng(1)
    x = np.exp2(r.uniform(-12, 8, size=20000))
    rel = 10.0 ** r.uniform(-8, -2, size=x.size)
    near, gap = B.near_boundary(x, rel)
    # brute force: rounding x moved by up to rel * x in either direction changes
    lo = O.e4m3_encode(x * (1 - rel))
    hi = O.e4m3_encode(x * (1 + rel))
    moved = lo != hi
    assert np.all(near[moved])                                   # every possible flip is flagged
    step = O.e4m3_decode(hi) - O.e4m3_decode(lo)
    assert np.all(step[moved] <= gap[moved] * (1 + 1e-12))


def _outlier_inputs(L, D, seed, outliers):
    r = np.random.default_rng(seed)
    x = [r.standard_normal((L, D)) for _ in range(3)]
    if outliers:
        cols = r.choice(D, 4, replace=False)
        for t in x:
            n = max(1, L * D // 1000)
            rr, cc = r.integers(0, L, n), cols[r.integers(0, 4, n)]
            t[rr, cc] = r.standard_normal(n) * 10
    x = [(t.astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)
         for t in x]
    return x, r.choice([-1.0, 1.0], size=D)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("outliers", [False, True])
def test_worst_bound_covers_the_emulation(causal, outliers):
    """The emulation is one rounding the GPU may produce: it lies within the
    worst-case bound of the exact attention of the dequantised inputs."""
    L, D = 600, 128
    (q, k, v), sigma = _outlier_inputs(L, D, 2 + causal, outliers)
    q8, qs, k8, ks, v8, vs = F.prepare_qkv(q, k, v, sigma)
    rows = np.arange(L)
    scale = D ** -0.5
    o, lse, tr = F.attention_fp8(q8, qs, k8, ks, v8, vs, rows, L, scale=scale, causal=causal, trace=True)
    tight, worst, amb = B.fp8_bounds(q8, qs, k8, ks, v8, vs, rows, L, scale=scale, causal=causal, o_emul=o,
                                     trace=tr)
    ox, _ = O.attention_head(F.dequantize(q8, qs), rows, F.dequantize(k8, ks), F.dequantize(v8, vs), L, scale,
                             causal)
    assert np.all(np.abs(o - ox) <= worst)
    assert amb.sum() <= 0.02 * L


@pytest.mark.parametrize("causal", [False, True])
def test_tight_bound_covers_perturbed_scores(causal):
    """Scores moved by a relative 2^-23 (inside the modelled fp32 error of
    each score) change only roundings within the tight bound."""
    L, D = 500, 128
    (q, k, v), sigma = _outlier_inputs(L, D, 7, True)
    q8, qs, k8, ks, v8, vs = F.prepare_qkv(q, k, v, sigma)
    rows = np.arange(L)
    scale = D ** -0.5
    o, lse, tr = F.attention_fp8(q8, qs, k8, ks, v8, vs, rows, L, scale=scale, causal=causal, trace=True)
    tight, _, amb = B.fp8_bounds(q8, qs, k8, ks, v8, vs, rows, L, scale=scale, causal=causal, o_emul=o,
                                 trace=tr, out_u=0.0)
    flips = 0
    for eps in (2.0 ** -23, -(2.0 ** -23)):
        o2, _, tr2 = F.attention_fp8(q8, qs, k8, ks, v8, vs, rows, L, scale=scale * (1 + eps), causal=causal,
                                     trace=True)
        d = np.abs(o2 - o)[~amb]
        assert np.all(d <= tight[~amb]), float((d / tight[~amb]).max())
        flips += sum(int((a["p8"] != b["p8"]).sum()) for a, b in zip(tr["tiles"], tr2["tiles"]))
    assert flips > 0          # the perturbation does move some roundings
