"""GPU parity of the attention backward (fa_bwd) through the C ABI against the
fp64 oracle's gradients.

The bar is an element-wise bound derived from the kernel's arithmetic (the
pages fix no tolerance for the backward). With u the unit roundoff of the
input type (2^-8 bf16, 2^-11 fp16), eps the relative error of the recomputed
P and n the length of each fp32 accumulation. eps comes from the forward's
stated LSE bar, not from the error this run happens to show: the test first
asserts |LSE - LSE_ref| <= 1e-3 for the LSE it passes in, and then takes
eps = expm1(1e-3) + 2^-18 (exp of an LSE off by at most 1e-3; the fp32
rounding of LSE log2 e and of the scaled score for |LSE| up to about 30, and
ex2.approx, stay under 2^-18):
  * O enters Delta rounded to 16 bits:   |dDelta_i| <= u sum_d |dO_id O_id|
  * dS = P (dP - Delta) rounded to 16 bits: |ddS_ij| <= (u + eps)|dS_ij| + P_ij |dDelta_i|
  * P rounded to 16 bits for dV:          (u + eps) P_ij
  * fp32 accumulation:                    n 2^-23 times the sum of |terms|
  * the output rounded to 16 bits:        u |result|
so, e.g., |dV_jd - ref| <= (u + eps + n 2^-23) (P^T |dO|)_jd + u |dV_jd|, and
dK, dQ carry the dS error through the products with |Q|, |K|. The test allows
twice the bound (plus 1e-6 absolute) at every element.
"""
import math

import numpy as np
import pytest
import torch

from exact_attention_forward_tiled_gb300 import api
from exact_attention_forward_tiled_gb300 import build as fa_build
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

U = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}
LSE_BAR = 1e-3                  # the forward's stated LSE tolerance
EPS = math.expm1(LSE_BAR) + 2.0 ** -18      # relative error of the recomputed P it allows


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    fa_build.build()
    api.lib()


def _rand(shape, dtype, seed, scale=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * scale).to(dtype)


def _bounds_head(q, k, v, do, o16, scale, causal, u, eps):
    """Element-wise error bounds of (dQ, dK, dV) for one (sequence, head)."""
    Lq, Lk = q.shape[0], k.shape[0]
    vis = orc._visible(Lq, Lk, causal)
    s = np.where(vis, scale * (q @ k.T), -np.inf)
    m = np.where(vis.any(axis=1), s.max(axis=1, initial=-np.inf, where=vis), 0.0)
    e = np.where(vis, np.exp(s - m[:, None]), 0.0)
    tot = e.sum(axis=1)
    p = np.divide(e, tot[:, None], out=np.zeros_like(e), where=tot[:, None] > 0)
    dp = do @ v.T
    ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
    ddelta = u * np.abs(do * o16).sum(axis=1)
    dds = (u + eps) * np.abs(ds) + p * ddelta[:, None]
    acc_q = Lk * 2.0 ** -23
    acc_k = Lq * 2.0 ** -23
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    dv = p.T @ do
    bq = scale * (dds @ np.abs(k)) + acc_q * scale * (np.abs(ds) @ np.abs(k)) + u * np.abs(dq)
    bk = scale * (dds.T @ np.abs(q)) + acc_k * scale * (np.abs(ds).T @ np.abs(q)) + u * np.abs(dk)
    bv = (u + eps + acc_k) * (p.T @ np.abs(do)) + u * np.abs(dv)
    return bq, bk, bv


def _check(B, H, Sq, Sk, D, causal, dtype, seed, lq=None, lk=None):
    varlen = lq is not None
    if varlen:
        B = len(lq)
        cq = torch.tensor(np.concatenate([[0], np.cumsum(lq)]), dtype=torch.int32, device="cuda")
        ck = torch.tensor(np.concatenate([[0], np.cumsum(lk)]), dtype=torch.int32, device="cuda")
        Tq, Tk = sum(lq), sum(lk)
        bq = [(int(cq[b]), int(cq[b + 1])) for b in range(B)]
        bk = [(int(ck[b]), int(ck[b + 1])) for b in range(B)]
    else:
        cq = ck = None
        Tq, Tk = B * Sq, B * Sk
        bq = [(b * Sq, (b + 1) * Sq) for b in range(B)]
        bk = [(b * Sk, (b + 1) * Sk) for b in range(B)]
    q = _rand((Tq, H, D), dtype, seed)
    k = _rand((Tk, H, D), dtype, seed + 1)
    v = _rand((Tk, H, D), dtype, seed + 2)
    do = _rand((Tq, H, D), dtype, seed + 3)
    scale = D ** -0.5
    kw = dict(cu_seqlens_q=cq, cu_seqlens_k=ck, max_seqlen_q=max(lq) if varlen else None,
              max_seqlen_k=max(lk) if varlen else None, batch=None if varlen else B)
    o, lse = api.attention_forward(q, k, v, causal=causal, scale=scale, **kw)
    dq, dk, dv = api.attention_backward(q, k, v, o, lse, do, causal=causal, scale=scale, **kw)
    api.fa_get_device_status()
    qn, kn, vn, don = (orc._f64(t.cpu()) for t in (q, k, v, do))
    o16 = orc._f64(o.cpu())
    rq, rk, rv = orc.attention_backward(qn, kn, vn, don, scale=scale, causal=causal, nseq=B, Sq=Sq, Sk=Sk,
                                        cu_seqlens_q=None if cq is None else cq.cpu().numpy(),
                                        cu_seqlens_k=None if ck is None else ck.cpu().numpy())
    _, lse_ref = orc.attention(qn, kn, vn, scale=scale, causal=causal, nseq=B, Sq=Sq, Sk=Sk,
                               cu_seqlens_q=None if cq is None else cq.cpu().numpy(),
                               cu_seqlens_k=None if ck is None else ck.cpu().numpy())
    l = lse.cpu().numpy()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(l), fin)
    assert (np.abs(l[fin] - lse_ref[fin]).max() if fin.any() else 0.0) <= LSE_BAR
    eps = EPS
    gq, gk, gv = (orc._f64(t.cpu()) for t in (dq, dk, dv))
    u = U[dtype]
    worst = 0.0
    for b in range(B):
        (qs, qe), (ks, ke) = bq[b], bk[b]
        for h in range(H):
            bnd = _bounds_head(qn[qs:qe, h], kn[ks:ke, h], vn[ks:ke, h], don[qs:qe, h], o16[qs:qe, h], scale,
                               causal, u, eps)
            for name, got, ref, bd in (("dQ", gq[qs:qe, h], rq[qs:qe, h], bnd[0]),
                                       ("dK", gk[ks:ke, h], rk[ks:ke, h], bnd[1]),
                                       ("dV", gv[ks:ke, h], rv[ks:ke, h], bnd[2])):
                if got.size == 0:
                    continue
                err = np.abs(got - ref)
                lim = 2.0 * bd + 1e-6
                ratio = (err / lim).max()
                worst = max(worst, ratio)
                assert ratio <= 1.0, (name, b, h, float(ratio), float(err.max()))
    return dq, dk, dv, worst


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Sq,Sk", [(128, 128), (300, 300), (256, 700), (700, 256), (1, 513), (129, 1)])
def test_backward_matches_oracle(D, causal, Sq, Sk):
    _check(2, 2, Sq, Sk, D, causal, torch.bfloat16, seed=Sq + 7 * Sk + D + causal)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_backward_fp16(D):
    _check(1, 3, 333, 520, D, True, torch.float16, seed=77 + D)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_backward_varlen(causal, D):
    _check(0, 2, 0, 0, D, causal, torch.bfloat16, seed=90 + D + causal, lq=[1, 300, 128, 0, 257, 40],
           lk=[129, 5, 400, 64, 0, 40])


@pytest.mark.parametrize("D", [128, 256])
def test_backward_is_deterministic(D):
    B, H, S = 2, 4, 640
    q, k, v, do = (_rand((B * S, H, D), torch.bfloat16, 200 + i) for i in range(4))
    o, lse = api.attention_forward(q, k, v, causal=True, batch=B)
    g1 = api.attention_backward(q, k, v, o, lse, do, causal=True, batch=B)
    g2 = api.attention_backward(q, k, v, o, lse, do, causal=True, batch=B)
    api.fa_get_device_status()
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_backward_no_keys_gives_zero_dq():
    """Sk = 0: the forward gives O = 0, LSE = -inf; every gradient is 0."""
    B, H, Sq, D = 2, 2, 200, 64
    q, do = _rand((B * Sq, H, D), torch.bfloat16, 300), _rand((B * Sq, H, D), torch.bfloat16, 301)
    k = torch.zeros((16, H, D), dtype=torch.bfloat16, device="cuda")   # never read: Sk = 0
    o = torch.zeros_like(q)
    lse = torch.full((B, H, Sq), float("-inf"), device="cuda")
    dq = torch.full_like(q, 7.0)
    dk = torch.empty_like(k)
    ws = torch.empty(api.fa_bwd_workspace_size(H, B * Sq), dtype=torch.uint8, device="cuda")
    api.fa_bwd(q, k, k, o, do, lse, dq, dk, dk, B, H, Sq, 0, D, 0.125, False, workspace=ws,
               workspace_bytes=ws.numel())
    api.fa_get_device_status()
    assert int(dq.abs().sum().item()) == 0


def _bounds_sampled(q, k, v, do, o16, lse_ref, rows, scale, causal, u, eps):
    """The element-wise bounds of ``_bounds_head`` at query rows ``rows`` (dQ)
    and key rows ``rows`` (dK, dV), from the oracle's LSE of the whole head."""
    Lq, Lk = q.shape[0], k.shape[0]
    lse_safe = np.where(np.isfinite(lse_ref), lse_ref, np.inf)
    ddelta = u * np.abs(do * o16).sum(axis=1)
    delta = (do * o16).sum(axis=1)      # magnitudes only; the 16-bit O is close enough here
    # rows of P (dQ)
    vr = orc._visible(Lq, Lk, causal, rows)
    pr = np.where(vr, np.exp(scale * (q[rows] @ k.T) - lse_safe[rows, None]), 0.0)
    dsr = pr * ((do[rows] @ v.T) - delta[rows, None])
    ddsr = (u + eps) * np.abs(dsr) + pr * ddelta[rows, None]
    dq = scale * (dsr @ k)
    bq = scale * (ddsr @ np.abs(k)) + Lk * 2.0 ** -23 * scale * (np.abs(dsr) @ np.abs(k)) + u * np.abs(dq)
    # columns of P (dK, dV)
    vc = orc._visible(Lq, Lk, causal)[:, rows]
    pc = np.where(vc, np.exp(scale * (q @ k[rows].T) - lse_safe[:, None]), 0.0)
    dsc = pc * ((do @ v[rows].T) - delta[:, None])
    ddsc = (u + eps) * np.abs(dsc) + pc * ddelta[:, None]
    dk = scale * (dsc.T @ q)
    dv = pc.T @ do
    bk = scale * (ddsc.T @ np.abs(q)) + Lq * 2.0 ** -23 * scale * (np.abs(dsc).T @ np.abs(q)) + u * np.abs(dk)
    bv = (u + eps + Lq * 2.0 ** -23) * (pc.T @ np.abs(do)) + u * np.abs(dv)
    return bq, bk, bv


@pytest.mark.parametrize("name", ["b1", "b2"])
def test_backward_full_size_sampled(name):
    """The backward workloads (bf16 D=128: B=4 H=16 S=8192 non-causal; B=2
    H=16 S=16384 causal), launched as the benchmark launches them, on sampled
    rows of two heads, with the same element-wise bound."""
    from exact_attention_forward_tiled_gb300 import workloads
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w, device="cuda")
    q, k, v, do = inp["q"], inp["k"], inp["v"], inp["do"]
    o, lse = api.attention_forward(q, k, v, causal=w.causal, batch=w.B)
    dq, dk, dv = api.attention_backward(q, k, v, o, lse, do, causal=w.causal, batch=w.B)
    api.fa_get_device_status()
    rng = np.random.default_rng(11)
    scale = w.D ** -0.5
    for b, h in ((0, 3), (w.B - 1, w.H - 1)):
        sl = slice(b * w.Sq, (b + 1) * w.Sq)
        qn, kn, vn, don = (orc._f64(t[sl, h].cpu()) for t in (q, k, v, do))
        o16 = orc._f64(o[sl, h].cpu())
        rows = np.concatenate([[0, 1, 127, 128, w.Sq - 1], rng.choice(np.arange(2, w.Sq - 1), 27, replace=False)])
        rq, rk, rv = orc.attention_backward_sampled(qn, kn, vn, don, rows, rows, scale=scale, causal=w.causal)
        _, lse_ref = orc.attention_head(qn, np.arange(w.Sq), kn, vn, w.Sq, scale, w.causal)
        l = lse[b, h].cpu().numpy()
        assert np.abs(l - lse_ref).max() <= LSE_BAR
        eps = EPS
        bnd = _bounds_sampled(qn, kn, vn, don, o16, lse_ref, rows, scale, w.causal, 2.0 ** -8, eps)
        for name, got, ref, bd in (("dQ", dq[sl, h][rows], rq, bnd[0]), ("dK", dk[sl, h][rows], rk, bnd[1]),
                                   ("dV", dv[sl, h][rows], rv, bnd[2])):
            err = np.abs(orc._f64(got.cpu()) - ref)
            ratio = (err / (2.0 * bd + 1e-6)).max()
            assert ratio <= 1.0, (name, b, h, float(ratio), float(err.max()))


@pytest.mark.parametrize("scale", [0.0, 1.0])
def test_backward_extreme_scales(scale):
    """scale 0: uniform P, dQ = dK = 0 and dV = the mean of dO; scale 1 at
    D = 128: a peaked softmax, where P and dS rounding matter most. Both
    under the element-wise bound."""
    B, H, S, D = 1, 2, 300, 128
    q, k, v, do = (_rand((B * S, H, D), torch.bfloat16, 400 + i) for i in range(4))
    o, lse = api.attention_forward(q, k, v, causal=True, scale=scale, batch=B)
    dq, dk, dv = api.attention_backward(q, k, v, o, lse, do, causal=True, scale=scale, batch=B)
    api.fa_get_device_status()
    qn, kn, vn, don = (orc._f64(t.cpu()) for t in (q, k, v, do))
    rq, rk, rv = orc.attention_backward(qn, kn, vn, don, scale=scale, causal=True, nseq=B, Sq=S, Sk=S)
    _, lse_ref = orc.attention(qn, kn, vn, scale=scale, causal=True, nseq=B, Sq=S, Sk=S)
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= LSE_BAR
    eps = EPS
    o16 = orc._f64(o.cpu())
    for h in range(H):
        bq, bk, bv = _bounds_head(qn[:, h], kn[:, h], vn[:, h], don[:, h], o16[:, h], scale, True, 2.0 ** -8, eps)
        for name, got, ref, bd in (("dQ", dq[:, h], rq[:, h], bq), ("dK", dk[:, h], rk[:, h], bk),
                                   ("dV", dv[:, h], rv[:, h], bv)):
            err = np.abs(orc._f64(got.cpu()) - ref)
            assert (err <= 2.0 * bd + 1e-6).all(), (name, h, float(err.max()))
    if scale == 0.0:
        assert int(dq.abs().sum().item()) == 0 and int(dk.abs().sum().item()) == 0


@pytest.mark.parametrize("seed", range(12))
def test_backward_random_shapes(seed):
    """Seeded draws of input type, head size, causal mask and fixed or varlen
    shapes (empty sequences included), every element within the bound."""
    r = np.random.default_rng(7000 + seed)
    dtype = [torch.float16, torch.bfloat16][r.integers(2)]
    D = int(r.choice([64, 128, 256]))
    causal = bool(r.integers(2))
    H = int(r.integers(1, 3))
    if r.integers(2):
        n = int(r.integers(1, 5))
        lq = [int(x) if r.random() > 0.15 else 0 for x in r.integers(1, 500, size=n)]
        lk = [int(x) if r.random() > 0.15 else 0 for x in r.integers(1, 500, size=n)]
        if sum(lq) == 0 or sum(lk) == 0:
            lq[0], lk[0] = 200, 137
        _check(None, H, max(lq), max(lk), D, causal, dtype, 7100 + 10 * seed, lq=lq, lk=lk)
    else:
        B = int(r.integers(1, 3))
        Sq, Sk = (int(x) for x in r.integers(1, 500, size=2))
        _check(B, H, Sq, Sk, D, causal, dtype, 7100 + 10 * seed)
