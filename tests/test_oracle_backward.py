"""Pins of the oracle's attention gradients (``attention_backward_head`` and
friends) to facts outside the function itself: central finite differences of
the C forward, closed forms, invariants; and plausible mistakes planted in a
copy of the function that the pins must catch.

The pages give no backward formula, so the gradient is the plain derivative
of the forward; finite differences of the (separately pinned) forward are the
independent route to it.
"""
import inspect
import textwrap

import numpy as np
import pytest

from oracle import oracle as orc

RNG = np.random.default_rng(20240611)


def _fwd_loss(q, k, v, do, scale, causal):
    """sum(O * dO): its gradient in (Q, K, V) is the backward of O for dO."""
    o, _ = orc.attention_head(q, np.arange(q.shape[0]), k, v, q.shape[0], scale, causal)
    return float((o * do).sum())


def _numeric_grads(q, k, v, do, scale, causal, h=1e-5):
    out = []
    for which in range(3):
        args = [q.copy(), k.copy(), v.copy()]
        x = args[which]
        g = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            x0 = x[idx]
            x[idx] = x0 + h
            fp = _fwd_loss(*args, do, scale, causal)
            x[idx] = x0 - h
            fm = _fwd_loss(*args, do, scale, causal)
            x[idx] = x0
            g[idx] = (fp - fm) / (2 * h)
        out.append(g)
    return out


def _rand(*shape):
    return RNG.standard_normal(shape)


# ------------------------------------------------------------------ pins
def pin_finite_differences(bwd):
    for Lq, Lk, causal in ((5, 7, False), (5, 7, True), (6, 3, True), (4, 4, True)):
        q, k, v, do = _rand(Lq, 4), _rand(Lk, 4), _rand(Lk, 4), _rand(Lq, 4)
        got = bwd(q, k, v, do, 0.7, causal)
        want = _numeric_grads(q, k, v, do, 0.7, causal)
        for g, w in zip(got, want):
            np.testing.assert_allclose(g, w, atol=1e-7, rtol=1e-6)


def pin_single_key(bwd):
    # one key: P = 1 for every row, so dQ = dK = 0 and dV = sum of the dO rows
    q, k, v, do = _rand(6, 8), _rand(1, 8), _rand(1, 8), _rand(6, 8)
    dq, dk, dv = bwd(q, k, v, do, 0.3, False)
    np.testing.assert_allclose(dq, 0, atol=1e-12)
    np.testing.assert_allclose(dk, 0, atol=1e-12)
    np.testing.assert_allclose(dv, do.sum(axis=0, keepdims=True), atol=1e-12)


def pin_zero_scale(bwd):
    # scale 0: P uniform 1 / Lk; dQ and dK carry the factor scale = 0
    q, k, v, do = _rand(5, 4), _rand(9, 4), _rand(9, 4), _rand(5, 4)
    dq, dk, dv = bwd(q, k, v, do, 0.0, False)
    np.testing.assert_allclose(dq, 0, atol=1e-12)
    np.testing.assert_allclose(dk, 0, atol=1e-12)
    np.testing.assert_allclose(dv, np.repeat(do.sum(axis=0, keepdims=True) / 9, 9, axis=0), atol=1e-12)


def pin_invariants(bwd):
    for causal in (False, True):
        Lq, Lk = 11, 8
        q, k, v, do = _rand(Lq, 6), _rand(Lk, 6), _rand(Lk, 6), _rand(Lq, 6)
        dq, dk, dv = bwd(q, k, v, do, 0.4, causal)
        # shifting every key by one vector leaves every softmax row unchanged
        np.testing.assert_allclose(dk.sum(axis=0), 0, atol=1e-10)
        # every row with a visible key spreads its dO over the keys with weights summing to 1
        seen = np.array([(not causal) or (i + Lk - Lq >= 0) for i in range(Lq)])
        np.testing.assert_allclose(dv.sum(axis=0), do[seen].sum(axis=0), atol=1e-10)
        # rows without a visible key get no gradient
        np.testing.assert_allclose(dq[~seen], 0, atol=1e-12)
        # linear in dO
        do2 = _rand(Lq, 6)
        g2 = bwd(q, k, v, do2, 0.4, causal)
        g3 = bwd(q, k, v, 2.0 * do - 3.0 * do2, 0.4, causal)
        for a, b, c in zip((dq, dk, dv), g2, g3):
            np.testing.assert_allclose(c, 2.0 * a - 3.0 * b, atol=1e-10)


BWD_PINS = [pin_finite_differences, pin_single_key, pin_zero_scale, pin_invariants]


@pytest.mark.parametrize("pin", BWD_PINS, ids=lambda p: p.__name__)
def test_backward_pins(pin):
    pin(orc.attention_backward_head)


def test_sampled_rows_equal_full_backward():
    for causal in (False, True):
        Lq, Lk, D = 37, 29, 8
        q, k, v, do = _rand(Lq, D), _rand(Lk, D), _rand(Lk, D), _rand(Lq, D)
        dq, dk, dv = orc.attention_backward_head(q, k, v, do, 0.35, causal)
        qr, kr = np.arange(Lq), np.arange(Lk)
        sq, sk, sv = orc.attention_backward_sampled(q, k, v, do, qr, kr, scale=0.35, causal=causal)
        np.testing.assert_allclose(sq, dq, atol=1e-11)
        np.testing.assert_allclose(sk, dk, atol=1e-11)
        np.testing.assert_allclose(sv, dv, atol=1e-11)


def test_packed_backward_is_per_sequence():
    H, D = 2, 4
    lq, lk = [3, 0, 5], [4, 2, 6]
    q, do = _rand(sum(lq), H, D), _rand(sum(lq), H, D)
    k, v = _rand(sum(lk), H, D), _rand(sum(lk), H, D)
    cq, ck = np.cumsum([0] + lq), np.cumsum([0] + lk)
    dq, dk, dv = orc.attention_backward(q, k, v, do, scale=0.5, causal=True, nseq=3, cu_seqlens_q=cq,
                                        cu_seqlens_k=ck)
    for b in range(3):
        for h in range(H):
            g = orc.attention_backward_head(q[cq[b]:cq[b + 1], h], k[ck[b]:ck[b + 1], h], v[ck[b]:ck[b + 1], h],
                                            do[cq[b]:cq[b + 1], h], 0.5, True)
            np.testing.assert_array_equal(g[0], dq[cq[b]:cq[b + 1], h])
            np.testing.assert_array_equal(g[1], dk[ck[b]:ck[b + 1], h])
            np.testing.assert_array_equal(g[2], dv[ck[b]:ck[b + 1], h])
    # keys of sequence 1 see no query: zero gradient
    np.testing.assert_array_equal(dk[4:6], 0)
    np.testing.assert_array_equal(dv[4:6], 0)


# ------------------------------------------------------------------ mutants
MUTANTS = {
    "dv_wrong_operand": ("dv = p.T @ do", "dv = p.T @ q"),
    "jacobian_term_dropped": ("ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))", "ds = p * dp"),
    "jacobian_sign": ("ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))",
                      "ds = p * (dp + (p * dp).sum(axis=1, keepdims=True))"),
    "jacobian_wrong_axis": ("ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))",
                            "ds = p * (dp - (p * dp).sum(axis=0, keepdims=True))"),
    "dq_scale_dropped": ("dq = scale * (ds @ k)", "dq = ds @ k"),
    "dq_uses_v": ("dq = scale * (ds @ k)", "dq = scale * (ds @ v)"),
    "dk_uses_do": ("dk = scale * (ds.T @ q)", "dk = scale * (ds.T @ do)"),
    "dp_uses_k": ("dp = do @ v.T", "dp = do @ k.T"),
    "causal_top_left": ("vis = _visible(Lq, Lk, causal)",
                        "vis = (_visible(Lq, Lq, causal)[:, :Lk] if Lk <= Lq else "
                        "np.pad(_visible(Lq, Lq, causal), ((0, 0), (0, Lk - Lq))))"),
    "softmax_over_columns": ("tot = e.sum(axis=1)", "tot = e.sum(axis=1) * 0 + e.sum()"),
}


def _mutant(name):
    old, new = MUTANTS[name]
    src = textwrap.dedent(inspect.getsource(orc.attention_backward_head))
    assert src.count(old) == 1, name
    ns = dict(vars(orc))
    exec(src.replace(old, new), ns)
    return ns["attention_backward_head"]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_backward_pins_catch_mutant(name):
    bwd = _mutant(name)
    caught = []
    for pin in BWD_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(bwd)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {name}"


def test_unmutated_copy_passes_every_pin():
    """The harness itself: the function re-created from its own source passes."""
    ns = dict(vars(orc))
    exec(textwrap.dedent(inspect.getsource(orc.attention_backward_head)), ns)
    for pin in BWD_PINS:
        pin(ns["attention_backward_head"])
