"""fp64 CPU oracle for exact tiled attention: the forward and its gradients.

TEST INFRASTRUCTURE ONLY. The only code that may import, call, link or run
anything in this package is the test suite (``tests/``), the smoke check in
``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py``. The GPU product path shares no code with this module and never
routes through it.

Every function cites the passage of the pages it follows. Page names:

* "FlashAttention-3 (lukebest wiki)" -- the FlashAttention-3 concept page,
  sections "3. FP8: throughput and precision" (block quantisation, incoherent
  processing).
* "Flash Attention 3 principles (guijiagi)" -- sections 1.2 (standard
  attention), 2.2 (online-softmax recurrence), 4.1.2 (E4M3 for the forward
  pass), 5.2 (varlen call with ``causal`` and ``softmax_scale``).

Parity status of each function (what pins it; see tests/test_oracle_*.py):

* ``attention`` -- pinned: torch's fp64 ``scaled_dot_product_attention`` and
  scipy's ``logsumexp`` (library routines), closed forms (single key, Q = 0,
  constant V), invariants (rows sum to 1, causal rows ignore future keys,
  key permutation, linearity in V, varlen packing).
* ``blockwise_attention`` -- pinned: equals ``attention`` by brute force over
  random block partitions (an independent algorithm, the pages' recurrence).
* ``hadamard`` / ``rotation`` -- pinned: ``scipy.linalg.hadamard``,
  H H^T = D I, M M^T = I, (QM)(KM)^T = QK^T.
* ``e4m3_encode`` / ``e4m3_decode`` -- pinned: exhaustive against torch's
  ``float8_e4m3fn`` casts.
* ``attention_backward_head`` / ``attention_backward`` -- pinned: central
  finite differences of the C forward (an independent route to the same
  derivative), closed forms (single key, scale = 0), invariants (dK rows sum
  to zero, dV rows sum to the dO rows, linearity in dO).
* ``attention_backward_sampled`` -- pinned: equals ``attention_backward_head``
  at every row on small inputs.
* ``attention_rows`` -- pinned: equals ``attention`` at the same rows, bit for
  bit (and shares its C core, which the mutant tests cover).
* ``merge_partials`` -- pinned: attention over disjoint key ranges, merged,
  equals attention over all keys from the definition; empty ranges merge to
  the other range (O = 0, LSE = -inf when every range is empty).
* ``visible_pairs`` -- pinned: brute-force counts of tiny causal and
  non-causal cases.
* ``e4m3_round`` -- decode of encode, both pinned above.

The FP8 path (Hadamard rotation, block quantisation, e4m3 attention) has its
own module, ``oracle/fp8.py``, with its parity status in its header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

E4M3_MAX = 448.0


# --------------------------------------------------------------------------
# build / load of the C core
# --------------------------------------------------------------------------
def build(force: bool = False) -> str:
    """Compile ``attention_oracle.c`` with gcc (OpenMP, no fast-math, no FMA
    contraction, so x86 and Arm give the same rounding)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.oracle_attention_rows.restype = ctypes.c_int
            lib.oracle_attention_rows.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_visible_pairs.restype = ctypes.c_int64
            lib.oracle_visible_pairs.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                                 ctypes.c_int64, ctypes.c_int]
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def _f64(x) -> np.ndarray:
    """Exact upcast of a torch tensor or array to a C-contiguous fp64 array."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu", torch.float64).contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _seq_bounds(nseq, Sq, Sk, cu_q, cu_k):
    if cu_q is None:
        bq = [(b * Sq, (b + 1) * Sq) for b in range(nseq)]
        bk = [(b * Sk, (b + 1) * Sk) for b in range(nseq)]
    else:
        cq = [int(c) for c in _as_list(cu_q)]
        ck = [int(c) for c in _as_list(cu_k)]
        bq = [(cq[b], cq[b + 1]) for b in range(nseq)]
        bk = [(ck[b], ck[b + 1]) for b in range(nseq)]
    return bq, bk


def _as_list(c):
    if hasattr(c, "detach"):
        return c.detach().cpu().tolist()
    return list(np.asarray(c).tolist())


# --------------------------------------------------------------------------
# exact attention (the plain definition)
# --------------------------------------------------------------------------
def attention_head(q_rows, qpos, k, v, Lq, scale, causal):
    """Attention of some query rows of one (sequence, head) pair.

    "Flash Attention 3 principles (guijiagi)" section 1.2 (S = QK^T,
    P = softmax(S), O = PV) with the softmax of section 2.2, the scale of the
    section 5.2 call and its causal mask (bottom-right aligned: row i sees
    keys j <= i + Lk - Lq). Returns (O [n, D], LSE [n]); LSE is the natural
    log of the sum of exp of the scaled scores.
    """
    lib = _load()
    q_rows = _f64(q_rows)
    k = _f64(k)
    v = _f64(v)
    qpos = np.ascontiguousarray(np.asarray(qpos, dtype=np.int64))
    n, D = q_rows.shape
    Lk = k.shape[0]
    o = np.empty((n, D), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = lib.oracle_attention_rows(q_rows.ctypes.data, qpos.ctypes.data, n,
                                   k.ctypes.data, v.ctypes.data, Lk, int(Lq), D,
                                   float(scale), int(bool(causal)),
                                   o.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise MemoryError("oracle_attention_rows failed")
    return o, lse


def attention(q, k, v, *, scale, causal, nseq, Sq=None, Sk=None,
              cu_seqlens_q=None, cu_seqlens_k=None):
    """Full attention forward over a packed ``[tokens, H, D]`` batch.

    Fixed length: ``nseq`` sequences of ``Sq`` query / ``Sk`` key rows, batch
    major. Varlen (section 5.2 of the guijiagi page): ``cu_seqlens_*`` are the
    prefix sums of the lengths. Returns (O fp64 ``[tokens, H, D]``,
    LSE fp64 ``[nseq, H, Sq]`` fixed or ``[H, total_q]`` varlen).
    """
    H, D = q.shape[1], q.shape[2]
    bq, bk = _seq_bounds(nseq, Sq, Sk, cu_seqlens_q, cu_seqlens_k)
    Tq = q.shape[0]
    o = np.zeros((Tq, H, D), dtype=np.float64)
    varlen = cu_seqlens_q is not None
    lse = np.zeros((H, Tq)) if varlen else np.zeros((nseq, H, Sq))
    for b in range(nseq):
        qs, qe = bq[b]
        ks, ke = bk[b]
        Lq = qe - qs
        if Lq == 0:
            continue
        for h in range(H):
            ob, lb = attention_head(q[qs:qe, h, :], np.arange(Lq), k[ks:ke, h, :], v[ks:ke, h, :],
                                    Lq, scale, causal)
            o[qs:qe, h, :] = ob
            if varlen:
                lse[h, qs:qe] = lb
            else:
                lse[b, h, :] = lb
    return o, lse


def attention_rows(q, k, v, rows, *, scale, causal, nseq, Sq=None, Sk=None,
                   cu_seqlens_q=None, cu_seqlens_k=None):
    """The same definition evaluated only at ``rows`` = [(seq, head, i), ...].

    Used for large problems where the full fp64 attention is too slow.
    Returns (O [n, D], LSE [n]) in the order of ``rows``.
    """
    bq, bk = _seq_bounds(nseq, Sq, Sk, cu_seqlens_q, cu_seqlens_k)
    rows = [tuple(int(x) for x in r) for r in rows]
    D = q.shape[2]
    o = np.zeros((len(rows), D))
    lse = np.zeros((len(rows),))
    groups = {}
    for idx, (b, h, i) in enumerate(rows):
        groups.setdefault((b, h), []).append((idx, i))
    for (b, h), items in groups.items():
        qs, qe = bq[b]
        ks, ke = bk[b]
        idxs = np.array([t[0] for t in items])
        pos = np.array([t[1] for t in items], dtype=np.int64)
        qsel = _f64(q[qs:qe, h, :])[pos]
        ob, lb = attention_head(qsel, pos, k[ks:ke, h, :], v[ks:ke, h, :], qe - qs, scale, causal)
        o[idxs] = ob
        lse[idxs] = lb
    return o, lse


def merge_partials(o_parts, lse_parts):
    """Combine attention over disjoint key ranges into attention over their
    union: LSE = ln sum_r exp(LSE_r), O = sum_r exp(LSE_r - LSE) O_r, where
    O_r is normalised over range r alone (the partial softmax of
    FlashDecoding, named in the "FlashAttention-3 (lukebest wiki)" lineage).
    o_parts [R, n, D], lse_parts [R, n]; a range with LSE_r = -inf carries no
    weight, and a row with no visible key at all gets O = 0, LSE = -inf."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = lse_parts.max(axis=0)
    o = np.zeros(o_parts.shape[1:])
    lse = np.full(lse_parts.shape[1:], -np.inf)
    ok = np.isfinite(m)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - np.where(ok, m, 0.0)), 0.0)
    tot = w.sum(axis=0)
    o[ok] = (w[:, ok, None] * o_parts[:, ok]).sum(axis=0) / tot[ok, None]
    lse[ok] = m[ok] + np.log(tot[ok])
    return o, lse


def visible_pairs(qpos, Lk, Lq, causal) -> int:
    """Number of (row, visible key) pairs of the given rows."""
    qpos = np.ascontiguousarray(np.asarray(qpos, dtype=np.int64))
    return int(_load().oracle_visible_pairs(qpos.ctypes.data, len(qpos), int(Lk), int(Lq), int(bool(causal))))


# --------------------------------------------------------------------------
# gradients of exact attention (the backward pass)
# --------------------------------------------------------------------------
def _visible(Lq, Lk, causal, qpos=None):
    """Boolean [n, Lk] mask of the keys each row sees (bottom-right aligned
    causal mask: row i sees keys j <= i + Lk - Lq)."""
    qpos = np.arange(Lq) if qpos is None else np.asarray(qpos, dtype=np.int64)
    j = np.arange(Lk)[None, :]
    if not causal:
        return np.ones((len(qpos), Lk), dtype=bool)
    return j <= qpos[:, None] + (Lk - Lq)


def attention_backward_head(q, k, v, do, scale, causal):
    """Gradients of one (sequence, head) pair: (dQ, dK, dV) in fp64.

    The pages print no backward formula ("FlashAttention-3 (lukebest wiki)"
    only reports its speed); this is the exact derivative of the forward of
    "Flash Attention 3 principles (guijiagi)" section 1.2 (S = scale QK^T
    with the section 5.2 causal mask, P = softmax(S) row by row, O = PV) for
    an upstream gradient dO, written out from the chain rule:

        dV = P^T dO
        dP = dO V^T
        dS_ij = P_ij (dP_ij - sum_l P_il dP_il)     (softmax Jacobian, row i)
        dQ = scale dS K,   dK = scale dS^T Q

    Masked pairs have P = 0 and so dS = 0; a row with no visible key has
    O = 0 and contributes nothing. Plain numpy on whole matrices.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    Lq, Lk = q.shape[0], k.shape[0]
    vis = _visible(Lq, Lk, causal)
    s = np.where(vis, scale * (q @ k.T), -np.inf)
    m = s.max(axis=1, initial=-np.inf, where=vis) if Lk else np.full(Lq, -np.inf)
    m = np.where(np.isfinite(m), m, 0.0)
    e = np.where(vis, np.exp(s - m[:, None]), 0.0)
    tot = e.sum(axis=1)
    p = np.divide(e, tot[:, None], out=np.zeros_like(e), where=tot[:, None] > 0)
    dv = p.T @ do
    dp = do @ v.T
    ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv


def attention_backward(q, k, v, do, *, scale, causal, nseq, Sq=None, Sk=None,
                       cu_seqlens_q=None, cu_seqlens_k=None):
    """``attention_backward_head`` over a packed ``[tokens, H, D]`` batch
    (fixed length or ``cu_seqlens`` packing, as ``attention``). Returns
    (dQ, dK, dV) fp64 with the shapes of q, k, v."""
    H = q.shape[1]
    bq, bk = _seq_bounds(nseq, Sq, Sk, cu_seqlens_q, cu_seqlens_k)
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    for b in range(nseq):
        qs, qe = bq[b]
        ks, ke = bk[b]
        for h in range(H):
            g = attention_backward_head(q[qs:qe, h], k[ks:ke, h], v[ks:ke, h], do[qs:qe, h], scale, causal)
            dq[qs:qe, h], dk[ks:ke, h], dv[ks:ke, h] = g
    return dq, dk, dv


def attention_backward_sampled(q, k, v, do, q_rows, k_rows, *, scale, causal):
    """Gradients of one (sequence, head) pair at some rows only, for problems
    too large for ``attention_backward_head``: dQ at query rows ``q_rows``,
    dK and dV at key rows ``k_rows``.

    Same definition, evaluated a row or a column of P at a time: the row
    normalisers LSE_i and O_i come from the C forward (``attention_head``),
    P_ij = exp(scale q_i.k_j - LSE_i) on visible pairs, and the Jacobian term
    sum_l P_il dP_il is taken as dO_i . O_i, which equals it exactly
    (sum_l P_il dO_i.v_l = dO_i . sum_l P_il v_l). Returns (dQ [nq, D],
    dK [nk, D], dV [nk, D]).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    Lq, Lk = q.shape[0], k.shape[0]
    o, lse = attention_head(q, np.arange(Lq), k, v, Lq, scale, causal)
    delta = (do * o).sum(axis=1)
    lse_safe = np.where(np.isfinite(lse), lse, np.inf)     # rows with no key: P = 0
    q_rows = np.asarray(q_rows, dtype=np.int64)
    k_rows = np.asarray(k_rows, dtype=np.int64)
    # rows of P for dQ
    vis = _visible(Lq, Lk, causal, q_rows)
    pr = np.where(vis, np.exp(scale * (q[q_rows] @ k.T) - lse_safe[q_rows, None]), 0.0)
    dsr = pr * ((do[q_rows] @ v.T) - delta[q_rows, None])
    dq = scale * (dsr @ k)
    # columns of P for dK, dV
    visc = _visible(Lq, Lk, causal)[:, k_rows]
    pc = np.where(visc, np.exp(scale * (q @ k[k_rows].T) - lse_safe[:, None]), 0.0)
    dsc = pc * ((do @ v[k_rows].T) - delta[:, None])
    dk = scale * (dsc.T @ q)
    dv = pc.T @ do
    return dq, dk, dv


# --------------------------------------------------------------------------
# the pages' blockwise recurrence, literally (cross-check of the definition)
# --------------------------------------------------------------------------
def blockwise_attention(q, k, v, block_edges, *, scale, causal=False):
    """Online softmax over key blocks, in the normalised form of
    "Flash Attention 3 principles (guijiagi)" section 2.2:

        m_new = max(m_old, m_j)
        l_new = l_old e^(m_old - m_new) + l_j e^(m_j - m_new)
        O_new = O_old (l_old e^(m_old - m_new)) / l_new + P_j V_j e^(m_j - m_new) / l_new

    with the symbols the page leaves undefined read as: m_j the row max of the
    block's scores S_j, P_j = exp(S_j - m_j), l_j the row sum of P_j.
    ``block_edges`` = sorted key indices [0, e1, ..., Lk] splitting the keys.
    One (sequence, head) pair, Lq = Lk alignment of the causal mask as in
    ``attention_head``. Returns (O, LSE) in fp64; pure numpy, tiny inputs only.
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    Lq, D = q.shape
    Lk = k.shape[0]
    o = np.zeros((Lq, D))
    lse = np.full((Lq,), -np.inf)
    for i in range(Lq):
        visible = Lk if not causal else min(Lk, i + Lk - Lq + 1)
        m_old, l_old, o_old = -np.inf, 0.0, np.zeros(D)
        for a, b in zip(block_edges[:-1], block_edges[1:]):
            b = min(b, visible)
            if b <= a:
                continue
            s_j = scale * (k[a:b] @ q[i])
            m_j = s_j.max()
            p_j = np.exp(s_j - m_j)
            l_j = p_j.sum()
            m_new = max(m_old, m_j)
            l_new = l_old * np.exp(m_old - m_new) + l_j * np.exp(m_j - m_new)
            o_old = (o_old * (l_old * np.exp(m_old - m_new)) / l_new
                     + (p_j @ v[a:b]) * np.exp(m_j - m_new) / l_new)
            m_old, l_old = m_new, l_new
        if l_old > 0:
            o[i] = o_old
            lse[i] = m_old + np.log(l_old)
    return o, lse


# --------------------------------------------------------------------------
# incoherent processing: Hadamard x random signs
# --------------------------------------------------------------------------
def hadamard(D: int) -> np.ndarray:
    """Sylvester Hadamard matrix of order D (a power of two), natural order:
    H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]]."""
    if D <= 0 or D & (D - 1):
        raise ValueError("D must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < D:
        h = np.block([[h, h], [h, -h]])
    return h


def rotation(sigma) -> np.ndarray:
    """M = diag(sigma) H_D / sqrt(D): the "Hadamard x +-1" orthogonal matrix of
    "FlashAttention-3 (lukebest wiki)" section 3 (incoherent processing), with
    the order and normalisation the page leaves open read as written here."""
    sigma = np.asarray(sigma, dtype=np.float64).reshape(-1)
    D = sigma.shape[0]
    return np.diag(sigma) @ hadamard(D) / np.sqrt(D)


# --------------------------------------------------------------------------
# E4M3 ("fn": no infinities, max +-448) codec, from the format definition
# --------------------------------------------------------------------------
def _e4m3_values() -> np.ndarray:
    vals = np.empty(256)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            vals[c] = np.nan
        elif e == 0:
            vals[c] = sign * m * 2.0 ** -9          # subnormal: (m/8) * 2^(1-7)
        else:
            vals[c] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


E4M3_VALUES = _e4m3_values()
_POS = E4M3_VALUES[:0x7F]   # codes 0x00..0x7E: 0 .. 448, increasing


def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3 code (uint8)."""
    return E4M3_VALUES[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(x) -> np.ndarray:
    """Round to nearest, ties to even, saturating to +-448 (E4M3 is the forward
    format, "Flash Attention 3 principles (guijiagi)" section 4.1.2). NaN maps
    to 0x7F. The sign of zero is kept."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    sign = np.signbit(x).astype(np.uint8) << 7
    hi = np.searchsorted(_POS, np.minimum(a, E4M3_MAX), side="left")
    hi = np.clip(hi, 0, len(_POS) - 1)
    lo = np.clip(hi - 1, 0, len(_POS) - 1)
    d_hi = np.abs(_POS[hi] - a)
    d_lo = np.abs(a - _POS[lo])
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(a >= E4M3_MAX, np.uint8(0x7E), code)
    code = (code | sign).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def e4m3_round(x) -> np.ndarray:
    """x rounded to the nearest E4M3 value (encode then decode)."""
    return e4m3_decode(e4m3_encode(x))
