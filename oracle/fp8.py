"""FP8 (e4m3) attention with per-tile block scales and Hadamard incoherent
processing, emulated on the CPU: the oracle of the FP8 path.

TEST INFRASTRUCTURE ONLY, under the same rule as the rest of ``oracle/``: only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import it. The GPU product path shares no code with it.

The method ("FlashAttention-3 (lukebest wiki)", technique 3, FP8 throughput
and precision): block quantisation, one scale per tile of 128 rows, and
incoherent processing, Q' = QM and K' = KM with M "Hadamard x random +-1",
orthogonal, so that Q'K'^T = QK^T while outlier features are spread over all
of D. "Flash Attention 3 principles (guijiagi)" section 4.1.2 picks E4M3 for
the forward pass.

Steps the pages leave open, read as follows (the CUDA path reads them the
same way):

* M = diag(sigma) H_D / sqrt(D), H_D the Sylvester Hadamard matrix in natural
  order, sigma in {+-1}^D; the same M for Q and K; V is not rotated.
* One fp32 scale per block of 128 rows of one (sequence, head), for each of
  Q', K' and V: amax / 448 of the block after the rotation (1 for an all-zero
  block); code = e4m3(x / scale), round to nearest even, saturating.
* The codes are integers decided by floating point, so they are decided in
  the kernel's precision, fp32, with every step correctly rounded: the
  rotation is the Walsh-Hadamard butterfly (strides 1, 2, ..., D/2) on
  sigma * x; 1/sqrt(D) is rounded once to fp32 and applied in the multiplier:
  scale = fp32(amax * norm) / 448, multiplier = norm / scale,
  code = e4m3(fp32(y * multiplier)).
* P becomes an e4m3 operand of the PV product. Keys are visited in tiles of
  128. The running max m_ref (log2 units) moves only when a tile's max exceeds
  it by more than tau = 4, and the accumulated O and l are rescaled when it
  does. Each P = 2^(s log2 e - m_ref) is rounded to e4m3 after being scaled by
  2^kappa v_s(j) / v_ref (kappa = 4; v_s(j) the V scale of key tile j, v_ref
  the largest V scale of the (sequence, head)), so x <= 2^(tau + kappa) = 256
  stays below 448, and multiplies the codes of V. l sums the unrounded P.
  O = v_ref 2^-kappa sum_j e4m3(x_j) v8_j / l; LSE = (m_ref + log2 l) ln 2.

Parity status: every function here is pinned in ``tests/test_oracle_fp8.py``
against routes other than itself (``scipy.linalg.hadamard``, torch's
``float8_e4m3fn`` casts, the fp64 definition of the rotation and the block
scales, the exact attention where every rounding is exact, hand-derived
closed forms), and ``tests/test_oracle_fp8_mutants.py`` plants plausible
mistakes in a copy of this file and checks that the pins catch each one.
"""
from __future__ import annotations

import numpy as np

from .oracle import E4M3_MAX, _f64, e4m3_decode, e4m3_encode

F32 = np.float32
TILE = 128          # rows per block scale and keys per tile
TAU = 4.0           # lazy-rescale threshold, log2 units
KAPPA = 4.0         # P is scaled by 2^kappa before it is rounded
LOG2E = 1.4426950408889634


def fwht(x, dtype=np.float64) -> np.ndarray:
    """x H_D for every row of x: the Walsh-Hadamard butterflies, strides 1, 2,
    ..., D/2, each add and subtract rounded in ``dtype``. H_D is symmetric, so
    this is also H_D applied to each row."""
    y = np.array(x, dtype=dtype)
    D = y.shape[-1]
    if D <= 0 or D & (D - 1):
        raise ValueError("D must be a power of two")
    lead = y.shape[:-1]
    h = 1
    while h < D:
        y = y.reshape(lead + (D // (2 * h), 2, h))
        a = y[..., 0, :].copy()
        b = y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        h *= 2
    return y.reshape(lead + (D,))


def rotation_norm(D: int) -> np.float32:
    """1/sqrt(D) rounded once to fp32."""
    return F32(1.0 / np.sqrt(D))


def prepare(x, sigma=None, block: int = TILE):
    """Block quantisation of one (sequence, head) [L, D] of 16-bit values,
    rotated by M = diag(sigma) H_D / sqrt(D) first when ``sigma`` is given.
    Returns (codes uint8 [L, D], scales fp32 [ceil(L / block)]), decided in
    fp32 as the module docstring states."""
    x32 = np.asarray(_f64(x), dtype=F32)
    L, D = x32.shape
    if sigma is not None:
        sg = np.asarray(_f64(sigma), dtype=F32).reshape(1, D)
        y = fwht(x32 * sg, F32)
        norm = rotation_norm(D)
    else:
        y = x32
        norm = F32(1.0)
    nb = (L + block - 1) // block
    codes = np.zeros((L, D), np.uint8)
    scales = np.ones(nb, F32)
    for b in range(nb):
        rows = slice(b * block, min((b + 1) * block, L))
        amax = F32(np.abs(y[rows]).max()) * norm
        s = amax / F32(E4M3_MAX) if amax > 0 else F32(1.0)
        mult = norm / s
        codes[rows] = e4m3_encode((y[rows] * mult).astype(F32))
        scales[b] = s
    return codes, scales


def prepare_qkv(q, k, v, sigma, block: int = TILE):
    """Q and K rotated by the same M and quantised; V quantised unrotated.
    Returns (q8, q_scale, k8, k_scale, v8, v_scale) of one (sequence, head)."""
    q8, qs = prepare(q, sigma, block)
    k8, ks = prepare(k, sigma, block)
    v8, vs = prepare(v, None, block)
    return q8, qs, k8, ks, v8, vs


def quantize_tensor(x, s):
    """Per-tensor FP8 (the comparison the wiki measures block quantisation
    against): codes e4m3(x / s) with one scale ``s`` for the whole tensor,
    no rotation, divided in fp64."""
    return e4m3_encode(_f64(x) / float(s))


def tensor_scale(x) -> float:
    """amax / 448 over a whole tensor (1 when it is all zero)."""
    amax = float(np.abs(_f64(x)).max()) if np.size(x) else 0.0
    return amax / E4M3_MAX if amax > 0 else 1.0


def dequantize(codes, scales, block: int = TILE) -> np.ndarray:
    """Real value of each code: code value times its block's scale."""
    val = e4m3_decode(codes)
    sc = np.repeat(np.asarray(scales, dtype=np.float64), block)[:val.shape[0]]
    return val * sc[:, None]


def attention_fp8(q8, q_scale, k8, k_scale, v8, v_scale, rows, Lq, *, scale, causal=False,
                  tau=TAU, kappa=KAPPA, block=TILE, trace=False):
    """O and LSE of the query positions ``rows`` of one (sequence, head) from
    the e4m3 codes and block scales of Q', K' and V, with P rounded to e4m3
    by the rule of the module docstring. Causal: row i sees key j when
    j <= i + Lk - Lq. Rows with no visible key get O = 0, LSE = -inf.

    With ``trace`` also returns, per key tile, the log2 scores ``t``, the
    visibility mask, the running max ``m_ref`` used for the tile, the
    previous one, the tile max, the unrounded ``x`` and the rounded ``p8``."""
    rows = np.asarray(rows, dtype=np.int64)
    q_val = dequantize(q8, q_scale, block)[rows]
    k_val = dequantize(k8, k_scale, block)
    v_code = e4m3_decode(v8)
    vs = np.asarray(v_scale, dtype=np.float64)
    Lk = k_val.shape[0]
    R, D = q_val.shape
    v_ref = float(vs.max()) if vs.size and vs.max() > 0 else 1.0
    lim = np.full(R, Lk, dtype=np.int64) if not causal else np.minimum(Lk, rows + Lk - Lq + 1)
    m_ref = np.full(R, -np.inf)
    l = np.zeros(R)
    acc = np.zeros((R, D))
    tiles = []
    for j in range((Lk + block - 1) // block):
        ks = slice(j * block, min((j + 1) * block, Lk))
        keys = np.arange(ks.start, ks.stop)
        vis = keys[None, :] < lim[:, None]
        t = np.where(vis, (scale * LOG2E) * (q_val @ k_val[ks].T), -np.inf)
        m_tile = t.max(axis=1)
        m_prev = m_ref.copy()
        if j == 0:
            m_ref = m_tile.copy()
        else:
            up = m_tile > m_ref + tau
            f = np.ones(R)
            f[up] = np.exp2(m_ref[up] - m_tile[up])      # 0 when m_ref is still -inf
            acc *= f[:, None]
            l *= f
            m_ref = np.where(up, m_tile, m_ref)
        m_safe = np.where(np.isfinite(m_ref), m_ref, 0.0)
        p = np.where(vis, np.exp2(np.where(vis, t, 0.0) - m_safe[:, None]), 0.0)
        x = p * (2.0 ** kappa * vs[j] / v_ref)
        p8 = e4m3_decode(e4m3_encode(x))
        acc += p8 @ v_code[ks]
        l += p.sum(axis=1)
        if trace:
            tiles.append({"j": j, "keys": ks, "t": t, "vis": vis, "m_ref": m_ref.copy(), "m_prev": m_prev,
                          "m_tile": m_tile, "x": x, "p8": p8})
    o = np.zeros((R, D))
    lse = np.full(R, -np.inf)
    ok = l > 0
    o[ok] = acc[ok] * (v_ref / (2.0 ** kappa * l[ok]))[:, None]
    lse[ok] = (m_ref[ok] + np.log2(l[ok])) * np.log(2.0)
    if trace:
        return o, lse, {"tiles": tiles, "v_ref": v_ref, "l": l, "m_ref": m_ref}
    return o, lse
