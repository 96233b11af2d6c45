"""Pins of the oracle's exact attention against things other than itself.

Each ``pin_*`` takes an ``att(q_rows, qpos, k, v, Lq, scale, causal) -> (O, LSE)``
callable with the signature of ``oracle.attention_head`` and raises
AssertionError when the callable disagrees with what the pages and the
mathematics fix. ``tests/test_oracle_attention.py`` runs them on the real
oracle; ``tests/test_oracle_mutants.py`` runs them on deliberately broken
copies of the oracle's C source to show that each plausible mistake trips at
least one pin.
"""
import math

import numpy as np
import scipy.special
import torch

TOL = 1e-12


def _rng(seed):
    return np.random.default_rng(seed)


def _full(att, q, k, v, scale, causal):
    Lq = q.shape[0]
    return att(q, np.arange(Lq), k, v, Lq, scale, causal)


def pin_sdpa(att):
    """torch's fp64 scaled_dot_product_attention (a library routine) agrees."""
    for seed, (L, D, causal) in enumerate([(1, 8, False), (7, 16, True), (64, 64, False),
                                           (130, 32, True), (33, 8, False)]):
        r = _rng(seed)
        q, k, v = (r.standard_normal((L, D)) for _ in range(3))
        scale = 0.3 + r.random()
        o, _ = _full(att, q, k, v, scale, causal)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q)[None, None], torch.from_numpy(k)[None, None],
            torch.from_numpy(v)[None, None], is_causal=causal, scale=scale)[0, 0].numpy()
        assert np.abs(o - ref).max() < 1e-11, ("sdpa", L, D, causal)


def pin_logsumexp(att):
    """LSE is scipy's logsumexp of the scaled visible scores (library routine)."""
    r = _rng(11)
    for causal in (False, True):
        L, D = 40, 16
        q, k, v = (r.standard_normal((L, D)) for _ in range(3))
        scale = 0.7
        _, lse = _full(att, q, k, v, scale, causal)
        s = scale * (q @ k.T)
        if causal:
            s = np.where(np.tril(np.ones((L, L), dtype=bool)), s, -np.inf)
        ref = scipy.special.logsumexp(s, axis=1)
        assert np.abs(lse - ref).max() < TOL, ("logsumexp", causal)


def pin_single_key(att):
    """One key: O = v_0 and LSE = scale * q . k_0 (closed form)."""
    r = _rng(3)
    D = 32
    q = r.standard_normal((5, D))
    k = r.standard_normal((1, D))
    v = r.standard_normal((1, D))
    o, lse = att(q, np.zeros(5, dtype=np.int64), k, v, 5, 0.25, False)
    assert np.abs(o - v[0]).max() < TOL
    assert np.abs(lse - 0.25 * (q @ k[0])).max() < TOL


def pin_rows_sum_to_one(att):
    """V = ones gives O = 1 for every row: the rows of P sum to 1."""
    r = _rng(4)
    for causal in (False, True):
        q, k = r.standard_normal((50, 24)), r.standard_normal((50, 24))
        o, _ = _full(att, q, k, np.ones((50, 24)), 1.3, causal)
        assert np.abs(o - 1.0).max() < TOL


def pin_constant_v(att):
    """Every value row equal to c gives O = c."""
    r = _rng(5)
    c = r.standard_normal(16)
    q, k = r.standard_normal((20, 16)), r.standard_normal((20, 16))
    o, _ = _full(att, q, k, np.tile(c, (20, 1)), 0.5, False)
    assert np.abs(o - c).max() < TOL


def pin_zero_q(att):
    """Q = 0: O is the mean of the visible V rows and LSE = ln |visible|;
    under the bottom-right causal mask row i of Lq sees i + Lk - Lq + 1 keys."""
    r = _rng(6)
    for Lq, Lk, causal in [(30, 30, False), (30, 30, True), (10, 25, True), (25, 10, True)]:
        D = 8
        q = np.zeros((Lq, D))
        k, v = r.standard_normal((Lk, D)), r.standard_normal((Lk, D))
        o, lse = att(q, np.arange(Lq), k, v, Lq, 0.9, causal)
        for i in range(Lq):
            n = Lk if not causal else min(Lk, i + Lk - Lq + 1)
            if n <= 0:
                assert np.all(o[i] == 0) and lse[i] == -np.inf, ("empty row", Lq, Lk, i)
            else:
                assert np.abs(o[i] - v[:n].mean(0)).max() < TOL, (Lq, Lk, i)
                assert abs(lse[i] - math.log(n)) < TOL, (Lq, Lk, i)


def pin_causal_ignores_future(att):
    """Causal: changing K/V rows j > i leaves row i bit-for-bit unchanged."""
    r = _rng(7)
    L, D = 40, 16
    q, k, v = (r.standard_normal((L, D)) for _ in range(3))
    o1, l1 = _full(att, q, k, v, 0.4, True)
    for cut in (0, 13, 39):
        k2, v2 = k.copy(), v.copy()
        k2[cut + 1:] += r.standard_normal(k2[cut + 1:].shape) * 5
        v2[cut + 1:] -= 3.0
        o2, l2 = _full(att, q, k2, v2, 0.4, True)
        assert np.array_equal(o1[:cut + 1], o2[:cut + 1]) and np.array_equal(l1[:cut + 1], l2[:cut + 1])


def pin_key_permutation(att):
    """Non-causal attention does not depend on the order of the keys."""
    r = _rng(8)
    q, k, v = r.standard_normal((9, 16)), r.standard_normal((31, 16)), r.standard_normal((31, 16))
    perm = r.permutation(31)
    o1, l1 = att(q, np.arange(9), k, v, 9, 0.6, False)
    o2, l2 = att(q, np.arange(9), k[perm], v[perm], 9, 0.6, False)
    assert np.abs(o1 - o2).max() < TOL and np.abs(l1 - l2).max() < TOL


def pin_linear_in_v(att):
    """O is linear in V: O(aV1 + bV2) = a O(V1) + b O(V2)."""
    r = _rng(9)
    q, k = r.standard_normal((12, 16)), r.standard_normal((12, 16))
    v1, v2 = r.standard_normal((12, 16)), r.standard_normal((12, 16))
    for causal in (False, True):
        oa, _ = _full(att, q, k, 2.5 * v1 - 0.75 * v2, 0.5, causal)
        o1, _ = _full(att, q, k, v1, 0.5, causal)
        o2, _ = _full(att, q, k, v2, 0.5, causal)
        assert np.abs(oa - (2.5 * o1 - 0.75 * o2)).max() < 1e-11


def pin_large_scores_stable(att):
    """Scores far outside exp's range still give the softmax (max subtraction):
    two keys with scores 1000 and 1000 - ln 3 weigh 3:1."""
    D = 4
    q = np.array([[1.0, 0, 0, 0]])
    k = np.array([[1000.0, 0, 0, 0], [1000.0 - math.log(3.0), 0, 0, 0]])
    v = np.array([[1.0, 0, 0, 0], [0, 1.0, 0, 0]])
    o, lse = att(q, np.zeros(1, dtype=np.int64), k, v, 1, 1.0, False)
    assert np.abs(o[0] - np.array([0.75, 0.25, 0, 0])).max() < TOL
    assert abs(lse[0] - (1000.0 + math.log(4.0 / 3.0))) < 1e-9


ALL_PINS = [pin_sdpa, pin_logsumexp, pin_single_key, pin_rows_sum_to_one, pin_constant_v,
            pin_zero_q, pin_causal_ignores_future, pin_key_permutation, pin_linear_in_v,
            pin_large_scores_stable]
