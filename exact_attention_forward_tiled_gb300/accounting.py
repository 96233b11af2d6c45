"""Work and traffic accounting for the attention forward (measurement only).

FLOP convention: 4 * Sq * Sk * D per (sequence, head) -- two matmuls, QK^T
and PV, of 2 * Sq * Sk * D each -- halved under the causal mask; varlen sums
4 * L_i^2 * D / 2 (causal) per sequence and head. Exponentials: Sq * Sk per
(sequence, head), halved under causal. The ratio FLOPs / exponentials = 4 D,
which is the 512x of the FlashAttention-3 essay (izhida) at head size 128.

Algorithmic bytes: one read of Q, K, V and one write of O and of the fp32
LSE; K/V re-reads across query tiles are served by L2 and are not counted.
"""
from __future__ import annotations

ELEM_BYTES = {"fp16": 2, "bf16": 2, "fp8": 1}


def attention_flops(H, D, lengths_q, lengths_k, causal) -> float:
    total = 0.0
    for lq, lk in zip(lengths_q, lengths_k):
        f = 4.0 * H * lq * lk * D
        total += f / 2 if causal else f
    return total


def visible_pair_flops(H, D, lengths_q, lengths_k, causal) -> float:
    """Forward FLOPs counted exactly, 4 * D per visible (query, key) pair, for
    workloads where Sq != Sk under the causal mask (bottom-right aligned:
    query i of Lq sees keys j <= i + Lk - Lq)."""
    total = 0
    for lq, lk in zip(lengths_q, lengths_k):
        if not causal:
            total += lq * lk
            continue
        # sum over i of clamp(i + lk - lq + 1, 0, lk)
        for i in range(lq):
            total += max(0, min(lk, i + lk - lq + 1))
    return 4.0 * H * D * total


def paged_kv_bytes(H, D, lengths_k, elem_bytes=2) -> float:
    """Algorithmic HBM bytes of a decode step over a paged cache: one read of
    every key and value row of every sequence."""
    return 2.0 * H * D * elem_bytes * sum(lengths_k)


def attention_bwd_flops(H, D, lengths_q, lengths_k, causal) -> float:
    """Backward FLOPs by the usual convention: five matrix products of
    2 * Sq * Sk * D each (S, dP, dV, dK, dQ), i.e. 2.5x the forward's, halved
    under the causal mask. Recomputation beyond them is not counted."""
    return 2.5 * attention_flops(H, D, lengths_q, lengths_k, causal)


def attention_exps(H, lengths_q, lengths_k, causal) -> float:
    total = 0.0
    for lq, lk in zip(lengths_q, lengths_k):
        e = float(H) * lq * lk
        total += e / 2 if causal else e
    return total


def attention_bytes(H, D, Tq, Tk, in_dtype, out_dtype="bf16", n_lse=None) -> float:
    """Algorithmic HBM bytes of one forward: read Q (Tq rows), K, V (Tk rows),
    write O (Tq rows) and LSE (fp32, one per query row and head)."""
    eb = ELEM_BYTES[in_dtype]
    ob = ELEM_BYTES[out_dtype]
    n_lse = Tq * H if n_lse is None else n_lse
    return H * D * (Tq * eb + 2 * Tk * eb + Tq * ob) + 4.0 * n_lse


def prep_bytes(H, D, B, S, in_dtype="bf16") -> float:
    """FP8 prep of Q, K, V (B sequences of S rows each): read three
    [B*S, H, D] 16-bit tensors, write three e4m3 tensors and three fp32 scale
    arrays (one per 128-row block of each (sequence, head))."""
    eb = ELEM_BYTES[in_dtype]
    nblk = B * ((S + 127) // 128)
    return 3.0 * (B * S * H * D * (eb + 1)) + 3.0 * 4 * H * nblk
