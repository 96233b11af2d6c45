"""Element-wise error bounds of the e4m3 attention, derived from its
arithmetic, for comparing the GPU's output with the FP8 oracle.

The GPU computes, per query row and 128-key tile (``oracle/fp8.py`` states
the rule): fp32 scores S = sum_d q8 k8 from exact e4m3 products, the log2
score t = S * c with c = scale * log2 e * q_s * k_s (rounded to fp32 in three
products), a lazy running max m_ref, x = ex2(t - m_ref + log2(2^kappa w_j)) in
fp32, P8 = e4m3(x), O_acc += P8 v8 (exact products, fp32 accumulation),
l += the unrounded x / (2^kappa w_j), and at the end O = O_acc v_ref / (2^kappa
l) rounded to bf16. Against the oracle, which evaluates the same rule in fp64:

* every non-flipped P8 is the same number; a P8 can only differ where x lies
  within the GPU's error of x (relative, ``rel``) of an e4m3 rounding
  boundary, and then by the gap between the two neighbours there;
* ``rel`` = ln 2 * delta, with delta (log2 units) summing the fp32
  accumulation of S (D + 2 roundings of sum |q8 k8|), the roundings of c
  and of the FMA, the same error in the tile max that sets m_ref, the error
  of lg2.approx in the V weight (2^-20 absolute, taken as a bound) and of
  ex2.approx (2^-21 relative, taken as a bound);
* the fp32 accumulation of O_acc: (keys + tiles + 4) u sum |P8 v8|;
* l: the largest ``rel`` of its terms plus (24 + 3 tiles) u + 2^-20;
* the final multiply and division: 3 u; the 16-bit output: u_out.

A row whose lazy-rescale decision (tile max > m_ref + tau) lies within the
GPU's error of the threshold may take the other branch, which changes the
rounding of every later P; such a row is "ambiguous" and is checked against
the exact attention of the dequantised inputs only, with the worst-case
bound: every P rounded by up to r(x) = min(1, max(2^-4, 2^-10 / x)) of
itself (e4m3 round to nearest: 2^-4 relative for normal x >= 2^-6, 2^-10
absolute below, everything under 2^-10 may become 0), where x is smallest
-- and r(x) largest -- when m_ref is the true row max.
"""
import math

import numpy as np

from oracle import oracle as O

U = 2.0 ** -24
LG2_ERR = 2.0 ** -20          # lg2.approx absolute error, log2 units (bound taken)
EX2_ERR = 2.0 ** -21          # ex2.approx relative error (bound taken)

_VALS = O.E4M3_VALUES[:0x7F]
_MIDS = (_VALS[:-1] + _VALS[1:]) / 2
_GAPS = np.diff(_VALS)


def e4m3_rel_err(x):
    """Largest relative rounding error of e4m3 round-to-nearest at x > 0."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.minimum(1.0, np.maximum(2.0 ** -4, np.where(x > 0, 2.0 ** -10 / x, np.inf)))


def near_boundary(x, rel):
    """(mask, gap): x within rel * x of an e4m3 rounding boundary, and the
    distance between the two e4m3 values on either side of it."""
    x = np.asarray(x, dtype=np.float64)
    i = np.clip(np.searchsorted(_MIDS, x), 1, len(_MIDS) - 1)
    d_lo, d_hi = np.abs(x - _MIDS[i - 1]), np.abs(_MIDS[i] - x)
    lo_closer = d_lo <= d_hi
    dist = np.where(lo_closer, d_lo, d_hi)
    gap = np.where(lo_closer, _GAPS[i - 1], _GAPS[i])
    return (dist <= rel * x) & (x > 0), gap


def fp8_bounds(q8, q_scale, k8, k_scale, v8, v_scale, rows, Lq, *, scale, causal, o_emul, trace,
               out_u=2.0 ** -8, tau=4.0, kappa=4.0, block=128):
    """Returns (tight [R, D], worst [R, D], ambiguous [R]):
    |O_gpu - o_emul| <= tight on rows that are not ambiguous, and
    |O_gpu - O_exact(dequantised)| <= worst on every row (module docstring)."""
    rows = np.asarray(rows, dtype=np.int64)
    qc = np.abs(O.e4m3_decode(q8))[rows]
    kc = np.abs(O.e4m3_decode(k8))
    vc = np.abs(O.e4m3_decode(v8))
    qs = np.asarray(q_scale, np.float64)[rows // block]
    ks = np.asarray(k_scale, np.float64)
    vs = np.asarray(v_scale, np.float64)
    R, D = qc.shape
    tiles = trace["tiles"]
    v_ref = trace["v_ref"]
    m_fin = trace["m_ref"]
    l_fin = trace["l"]
    c_row = scale * math.log2(math.e) * qs
    # S error of every visible pair and its largest value per row (the tile
    # max and hence m_ref carry at most that much)
    d_s = []
    d_max = np.zeros(R)
    for tl in tiles:
        ksl = tl["keys"]
        ds = (D + 2) * U * (qc @ kc[ksl].T) * (c_row[:, None] * ks[tl["j"]]) + 4 * U * np.where(
            tl["vis"], np.abs(np.where(tl["vis"], tl["t"], 0.0)), 0.0)
        ds = np.where(tl["vis"], ds, 0.0)
        d_s.append(ds)
        d_max = np.maximum(d_max, ds.max(axis=1))
    m_true = np.max([np.where(tl["vis"], tl["t"], -np.inf).max(axis=1) for tl in tiles], axis=0)
    with np.errstate(invalid="ignore"):
        fin = np.where(np.isfinite(m_fin), m_fin, 0.0)
    ambiguous = np.zeros(R, dtype=bool)
    flip = np.zeros((R, D))
    acc_abs = np.zeros((R, D))
    worst_p = np.zeros((R, D))
    rel_max = np.zeros(R)
    n_keys = np.zeros(R)
    p_sum = np.zeros(R)
    for tl, ds in zip(tiles, d_s):
        ksl, vis, t, x, p8 = tl["keys"], tl["vis"], tl["t"], tl["x"], tl["p8"]
        m_ref = np.where(np.isfinite(tl["m_ref"]), tl["m_ref"], 0.0)
        if tl["j"] > 0:
            m_prev, m_tile = tl["m_prev"], tl["m_tile"]
            both = np.isfinite(m_prev) & np.isfinite(m_tile)
            margin = np.full(R, np.inf)
            margin[both] = np.abs(m_tile[both] - m_prev[both] - tau)
            ambiguous |= margin <= 2 * d_max + 8 * U * (np.abs(np.where(both, m_tile, 0.0)) + tau + 16)
        tt = np.where(vis, t, 0.0)
        delta = ds + d_max[:, None] + LG2_ERR + EX2_ERR / math.log(2.0) + 4 * U * (np.abs(tt) + np.abs(m_ref)[:, None] + 16)
        rel = np.expm1(math.log(2.0) * delta) * 1.01
        rel = np.where(vis, rel, 0.0)
        rel_max = np.maximum(rel_max, rel.max(axis=1))
        near, gap = near_boundary(x, rel)
        # contributions in units of the final m_ref
        f = np.exp2(np.where(np.isfinite(tl["m_ref"]), m_ref - fin, 0.0))[:, None]
        flip += f * ((near & vis) * gap) @ vc[ksl]
        acc_abs += f * p8 @ vc[ksl]
        n_keys += vis.sum(axis=1)
        # worst case against the exact attention: P relative to the true max
        w = vs[tl["j"]] / v_ref
        with np.errstate(invalid="ignore", over="ignore"):
            p_true = np.where(vis, np.exp2(tt - np.where(np.isfinite(m_true), m_true, 0.0)[:, None]), 0.0)
        x0 = p_true * (2.0 ** kappa * w)
        worst_p += (e4m3_rel_err(x0) * (1 + rel) * p_true) @ (vc[ksl] * vs[tl["j"]])
        p_sum += p_true.sum(axis=1)
    n_tiles = len(tiles)
    ok = l_fin > 0
    scale_o = np.where(ok, v_ref / (2.0 ** kappa * np.where(ok, l_fin, 1.0)), 0.0)[:, None]
    gamma = ((n_keys + n_tiles + 4) * U)[:, None]
    eps_l = (rel_max + (24 + 3 * n_tiles) * U + LG2_ERR)[:, None]
    o_abs = np.abs(o_emul)
    t_acc = scale_o * gamma * acc_abs
    tight_t = scale_o * flip + t_acc + (eps_l + 3 * U) * o_abs
    tight = out_u * (o_abs + tight_t) + tight_t + 1e-30
    worst_t = np.where(p_sum > 0, 1.0 / np.where(p_sum > 0, p_sum, 1.0), 0.0)[:, None] * worst_p
    worst_t = worst_t + tight_t
    # |O_exact| <= |o_emul| + worst_t bounds the magnitude the output rounds
    worst = out_u * (o_abs + 2 * worst_t) + worst_t + 1e-30
    return tight, worst, ambiguous


def check_attention(o_gpu, lse_gpu, q8, q_scale, k8, k_scale, v8, v_scale, rows, Lq, *, scale, causal,
                    out_u=2.0 ** -8, lse_tol=1e-3):
    """Compare the GPU's O and LSE rows of one (sequence, head) with the FP8
    oracle element by element: within twice the tight bound of the emulation
    on every row that is not ambiguous, within twice the worst-case bound of
    the exact attention of the dequantised inputs on every row, and LSE within
    ``lse_tol`` of both (they are the same number: l sums the unrounded P).
    Returns a dict of the largest error-to-bound ratios and the counts."""
    from oracle import fp8 as F
    rows = np.asarray(rows, dtype=np.int64)
    o_e, lse_e, tr = F.attention_fp8(q8, q_scale, k8, k_scale, v8, v_scale, rows, Lq, scale=scale,
                                     causal=causal, trace=True)
    tight, worst, amb = fp8_bounds(q8, q_scale, k8, k_scale, v8, v_scale, rows, Lq, scale=scale, causal=causal,
                                   o_emul=o_e, trace=tr, out_u=out_u)
    qd, kd, vd = F.dequantize(q8, q_scale), F.dequantize(k8, k_scale), F.dequantize(v8, v_scale)
    o_x, lse_x = O.attention_head(qd[rows], rows, kd, vd, Lq, scale, causal)
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    err_e = np.abs(o_gpu - o_e)
    err_x = np.abs(o_gpu - o_x)
    r_tight = float((err_e / tight)[~amb].max()) if (~amb).any() else 0.0
    r_worst = float((err_x / worst).max()) if err_x.size else 0.0
    assert r_tight <= 2.0, ("GPU O outside twice the tight bound of the emulation", r_tight)
    assert r_worst <= 2.0, ("GPU O outside twice the worst-case bound of the exact attention", r_worst)
    fin = np.isfinite(lse_e)
    assert np.array_equal(np.isfinite(lse_gpu), fin)
    assert np.abs(lse_e[fin] - lse_x[fin]).max(initial=0.0) <= 1e-9
    d_lse = float(np.abs(lse_gpu[fin] - lse_e[fin]).max(initial=0.0))
    assert d_lse <= lse_tol, d_lse
    return {"ratio_tight": r_tight, "ratio_worst": r_worst, "ambiguous": int(amb.sum()), "rows": len(rows),
            "max_err_emul": float(err_e.max(initial=0.0)), "max_err_exact": float(err_x.max(initial=0.0)),
            "lse": d_lse}
