"""CPU tests of the fp64 oracle's exact attention and the pages' recurrence."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests.oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pins(pin):
    pin(O.attention_head)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L,D", [(1, 8), (17, 16), (96, 32), (130, 64)])
def test_blockwise_recurrence_equals_direct(L, D, causal):
    """The pages' online-softmax recurrence (normalised form) reaches the
    direct softmax for random partitions of the keys into blocks."""
    r = np.random.default_rng(L * 7 + D + causal)
    q, k, v = (r.standard_normal((L, D)) for _ in range(3))
    o_ref, lse_ref = O.attention_head(q, np.arange(L), k, v, L, 0.37, causal)
    for trial in range(4):
        cuts = sorted(set(r.integers(1, max(L, 2), size=r.integers(0, 6)).tolist()))
        edges = [0] + [c for c in cuts if 0 < c < L] + [L]
        o, lse = O.blockwise_attention(q, k, v, edges, scale=0.37, causal=causal)
        assert np.abs(o - o_ref).max() < 1e-12
        assert np.abs(lse - lse_ref).max() < 1e-12


def test_varlen_equals_per_sequence():
    """Packing sequences with cu_seqlens changes nothing: every sequence
    equals its own fixed-length attention, whatever the other sequences hold."""
    r = np.random.default_rng(21)
    lens = [5, 1, 37, 12]
    H, D = 3, 16
    T = sum(lens)
    q, k, v = (r.standard_normal((T, H, D)) for _ in range(3))
    cu = np.concatenate([[0], np.cumsum(lens)])
    for causal in (False, True):
        o, lse = O.attention(q, k, v, scale=0.5, causal=causal, nseq=len(lens),
                             cu_seqlens_q=cu, cu_seqlens_k=cu)
        for b, L in enumerate(lens):
            s, e = cu[b], cu[b + 1]
            ob, lb = O.attention(q[s:e], k[s:e], v[s:e], scale=0.5, causal=causal, nseq=1, Sq=L, Sk=L)
            assert np.array_equal(o[s:e], ob)
            assert np.array_equal(lse[:, s:e], lb[0])
        k2 = k.copy()
        k2[cu[2]:cu[3]] += 7.0   # disturb sequence 2 only
        o2, _ = O.attention(q, k2, v, scale=0.5, causal=causal, nseq=len(lens),
                            cu_seqlens_q=cu, cu_seqlens_k=cu)
        assert np.array_equal(o2[:cu[2]], o[:cu[2]]) and np.array_equal(o2[cu[3]:], o[cu[3]:])


def test_rows_equal_full():
    r = np.random.default_rng(22)
    B, S, H, D = 2, 40, 2, 16
    q, k, v = (torch.from_numpy(r.standard_normal((B * S, H, D))).to(torch.bfloat16) for _ in range(3))
    o, lse = O.attention(q, k, v, scale=0.25, causal=True, nseq=B, Sq=S, Sk=S)
    rows = [(0, 0, 0), (1, 1, 39), (0, 1, 17), (1, 0, 3)]
    orow, lrow = O.attention_rows(q, k, v, rows, scale=0.25, causal=True, nseq=B, Sq=S, Sk=S)
    for n, (b, h, i) in enumerate(rows):
        assert np.array_equal(orow[n], o[b * S + i, h])
        assert lrow[n] == lse[b, h, i]


def test_scale_folds_into_q():
    """scale * (q . k) == (scale * q) . k up to fp64 rounding."""
    r = np.random.default_rng(23)
    q, k, v = (r.standard_normal((20, 32)) for _ in range(3))
    a = O.attention_head(q, np.arange(20), k, v, 20, 0.125, False)
    b = O.attention_head(q * 0.125, np.arange(20), k, v, 20, 1.0, False)
    assert np.abs(a[0] - b[0]).max() < 1e-12 and np.abs(a[1] - b[1]).max() < 1e-12


def test_visible_pairs():
    assert O.visible_pairs(np.arange(4), 4, 4, False) == 16
    assert O.visible_pairs(np.arange(4), 4, 4, True) == 10
    assert O.visible_pairs(np.arange(2), 5, 2, True) == 4 + 5
    assert O.visible_pairs(np.arange(3), 1, 3, True) == 1


def test_pages_numbers():
    """Numbers the pages print that pin the measurement conventions."""
    from exact_attention_forward_tiled_gb300 import accounting as A
    with open(os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")) as f:
        g = json.load(f)
    # matmul FLOPs per exponential at head size 128 (izhida essay, MUFU paragraph)
    e = g["matmul_flops_per_exp_hdim128"]
    D = 128
    assert A.attention_flops(1, D, [300], [300], False) / A.attention_exps(1, [300], [300], False) == e["value"]
    assert A.attention_flops(1, D, [300], [300], True) / A.attention_exps(1, [300], [300], True) == e["value"]
    # exp time relative to matmul time on H100 from the same paragraph's
    # throughputs: (989 / 3.9) / 512 ~ 0.5, the "about 50%" of its arithmetic
    t = g["h100_fp16_matmul_vs_mufu_tflops"]
    ratio = (t["matmul"] / t["mufu"]) / e["value"]
    assert abs(ratio - g["exp_time_fraction_of_matmul"]["value"]) < 0.01


@pytest.mark.parametrize("cuts", [[0, 40], [0, 1, 2, 97], [0, 30, 31, 60, 120]])
def test_merge_of_key_ranges_equals_full(cuts):
    """Attention over disjoint key ranges, merged, is attention over all keys
    (the identity split-KV relies on); pinned against the direct definition."""
    r = np.random.default_rng(len(cuts))
    Lq, Lk, D = 17, 120, 32
    q, k, v = r.standard_normal((Lq, D)), r.standard_normal((Lk, D)), r.standard_normal((Lk, D))
    edges = cuts + [Lk]
    parts = [O.attention_head(q, np.arange(Lq), k[a:b], v[a:b], Lq, 0.3, False)
             for a, b in zip(edges[:-1], edges[1:])]
    o, lse = O.merge_partials([p[0] for p in parts], [p[1] for p in parts])
    o_ref, lse_ref = O.attention_head(q, np.arange(Lq), k, v, Lq, 0.3, False)
    assert np.abs(o - o_ref).max() < 1e-12 and np.abs(lse - lse_ref).max() < 1e-12


def test_merge_handles_empty_ranges():
    o1 = np.array([[1.0, 2.0], [0.0, 0.0]])
    l1 = np.array([0.5, -np.inf])
    o2 = np.zeros((2, 2))
    l2 = np.array([-np.inf, -np.inf])
    o, lse = O.merge_partials([o1, o2], [l1, l2])
    assert np.array_equal(o[0], o1[0]) and lse[0] == 0.5
    assert np.all(o[1] == 0) and lse[1] == -np.inf
