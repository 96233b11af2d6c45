"""GPU parity of the CUDA attention forward against the fp64 oracle, through the
C ABI. Tolerances (written here, from the stated bars): max |O - O_ref| <= 2e-3
for fp16 inputs, <= 1e-2 for bf16; max |LSE - LSE_ref| <= 1e-3."""
import numpy as np
import pytest
import torch

from exact_attention_forward_tiled_gb300 import api, workloads
from exact_attention_forward_tiled_gb300 import build as fa_build
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

TOL_O = {torch.float16: 2e-3, torch.bfloat16: 1e-2}
TOL_LSE = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    fa_build.build()
    api.lib()


def _rand(shape, dtype, seed, scale=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * scale).to(dtype)


def _run(q, k, v, **kw):
    o, lse = api.attention_forward(q, k, v, **kw)
    api.fa_get_device_status()
    return o, lse


def _check(o, lse, o_ref, lse_ref, dtype, what, tol_o=None):
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    err_o = np.abs(o - o_ref).max() if o.size else 0.0
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: -inf pattern of LSE differs"
    err_l = np.abs(lse[fin] - lse_ref[fin]).max() if fin.any() else 0.0
    tol_o = TOL_O[dtype] if tol_o is None else tol_o
    assert err_o <= tol_o, f"{what}: max|dO| = {err_o:.3e} > {tol_o:.3e}"
    assert err_l <= TOL_LSE, f"{what}: max|dLSE| = {err_l:.3e}"
    return err_o, err_l


def _fixed(B, H, Sq, Sk, D, causal, dtype, seed, scale=None):
    q = _rand((B * Sq, H, D), dtype, seed)
    k = _rand((B * Sk, H, D), dtype, seed + 1)
    v = _rand((B * Sk, H, D), dtype, seed + 2)
    scale = D ** -0.5 if scale is None else scale
    o, lse = _run(q, k, v, causal=causal, scale=scale, batch=B)
    o_ref, lse_ref = orc.attention(q.cpu(), k.cpu(), v.cpu(), scale=scale, causal=causal, nseq=B,
                                   Sq=Sq, Sk=Sk)
    return _check(o, lse, o_ref, lse_ref, dtype, f"B{B} H{H} Sq{Sq} Sk{Sk} D{D} causal={causal}")


def test_c1_full():
    """fp16, B=1, H=2, Sq=Sk=256, D=64, non-causal, seed 0: every element."""
    w = workloads.WORKLOADS["c1"]
    inp = workloads.make_inputs(w, device="cuda")
    q, k, v = inp["q"], inp["k"], inp["v"]
    o, lse = _run(q, k, v, causal=False, scale=w.D ** -0.5, batch=w.B)
    o_ref, lse_ref = orc.attention(q.cpu(), k.cpu(), v.cpu(), scale=w.D ** -0.5, causal=False,
                                   nseq=w.B, Sq=w.Sq, Sk=w.Sk)
    _check(o, lse, o_ref, lse_ref, torch.float16, "c1")


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("S", [1, 127, 128, 129, 255, 257])
@pytest.mark.parametrize("causal", [False, True])
def test_edge_lengths(D, S, causal):
    dtype = torch.float16 if D == 64 else torch.bfloat16
    _fixed(2, 3, S, S, D, causal, dtype, seed=D + S + causal)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("Sq,Sk", [(100, 300), (300, 100), (384, 640), (1, 513)])
@pytest.mark.parametrize("causal", [False, True])
def test_unequal_lengths(D, Sq, Sk, causal):
    """Sq != Sk: the causal mask is bottom-right aligned; rows that see no key
    give O = 0 and LSE = -inf."""
    _fixed(2, 2, Sq, Sk, D, causal, torch.bfloat16, seed=7 * D + Sq + Sk)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_longer_multi_tile(dtype):
    _fixed(1, 2, 1024 + 77, 1024 + 77, 128, True, dtype, seed=3)
    _fixed(1, 2, 1024, 2048 + 5, 128, False, dtype, seed=4)


def test_scale_values():
    for scale in (0.0, 0.01, 1.0):
        _fixed(1, 2, 200, 200, 64, False, torch.float16, seed=11, scale=scale)


def test_large_scores_trigger_rescale():
    """Scores that grow along the keys force the lazy rescale of O many times.

    The softmax here is peaked, so |O| reaches max |V| (~4.5) instead of the
    ~0.02 of the N(0,1) workloads, and the absolute 1e-2 bar is below what a
    bf16 pipeline resolves at that magnitude: P rounded to bf16 (unit
    roundoff u = 2^-8) moves O by up to u * max|V| and the bf16 output by up
    to u * |O|. The bar is therefore 2 u max|V| + 1e-2."""
    B, H, S, D = 1, 2, 1024, 128
    q = _rand((S, H, D), torch.bfloat16, 21)
    k = _rand((S, H, D), torch.bfloat16, 22)
    ramp = torch.linspace(0.1, 6.0, S, device="cuda").view(S, 1, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    q = (q.float() * 3).to(torch.bfloat16)
    v = _rand((S, H, D), torch.bfloat16, 23)
    for causal in (False, True):
        o, lse = _run(q, k, v, causal=causal, scale=D ** -0.5, batch=B)
        o_ref, lse_ref = orc.attention(q.cpu(), k.cpu(), v.cpu(), scale=D ** -0.5, causal=causal,
                                       nseq=B, Sq=S, Sk=S)
        tol = 2 * 2.0 ** -8 * v.float().abs().max().item() + 1e-2
        _check(o, lse, o_ref, lse_ref, torch.bfloat16, f"ramp causal={causal}", tol_o=tol)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_small(D, causal):
    lens = [1, 127, 128, 129, 300, 5, 0, 513, 256]
    H = 2
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device="cuda")
    T = int(cu[-1])
    dtype = torch.bfloat16
    q, k, v = (_rand((T, H, D), dtype, 100 + i + D) for i in range(3))
    o, lse = _run(q, k, v, causal=causal, scale=D ** -0.5, cu_seqlens_q=cu, cu_seqlens_k=cu,
                  max_seqlen_q=max(lens), max_seqlen_k=max(lens))
    o_ref, lse_ref = orc.attention(q.cpu(), k.cpu(), v.cpu(), scale=D ** -0.5, causal=causal,
                                   nseq=len(lens), cu_seqlens_q=cu.cpu(), cu_seqlens_k=cu.cpu())
    _check(o, lse, o_ref, lse_ref, dtype, f"varlen D{D} causal={causal}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_runs_of_empty_tiles(D, causal):
    """One long sequence among many one-token ones: most work tiles (the query
    blocks a short sequence does not have) are empty, in runs longer than the
    tile ring is deep, so every role must pass them without waiting on one
    another. Every row against the oracle, and no device status raised."""
    lens = [1] * 20 + [3000] + [1] * 20 + [200]
    H = 4
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device="cuda")
    T = int(cu[-1])
    dtype = torch.bfloat16
    q, k, v = (_rand((T, H, D), dtype, 900 + i + D) for i in range(3))
    o, lse = _run(q, k, v, causal=causal, scale=D ** -0.5, cu_seqlens_q=cu, cu_seqlens_k=cu,
                  max_seqlen_q=max(lens), max_seqlen_k=max(lens))
    o_ref, lse_ref = orc.attention(q.cpu(), k.cpu(), v.cpu(), scale=D ** -0.5, causal=causal,
                                   nseq=len(lens), cu_seqlens_q=cu.cpu(), cu_seqlens_k=cu.cpu())
    _check(o, lse, o_ref, lse_ref, dtype, f"varlen empty runs D{D} causal={causal}")


def test_varlen_bad_seqlens_reported():
    """A cu_seqlens entry beyond total_q is caught by the kernel's own bounds
    check: the sequence is skipped and the status word reports it."""
    H, D = 2, 64
    q, k, v = (_rand((256, H, D), torch.bfloat16, 200 + i) for i in range(3))
    cu = torch.tensor([0, 128, 512], dtype=torch.int32, device="cuda")  # 512 > 256 rows
    o = torch.zeros_like(q)
    lse = torch.zeros((H, 256), device="cuda")
    api.fa_fwd(q, k, v, o, lse, 2, H, 384, 384, D, 0.125, 0, cu, cu, 256, 256)
    st, raw = api.fa_get_device_status(check=False)
    assert st == -6, (st, hex(raw))
    assert api.fa_get_device_status(check=False)[0] == 0      # read-and-clear
    o_ref, _ = orc.attention(q[:128].cpu(), k[:128].cpu(), v[:128].cpu(), scale=0.125, causal=False,
                             nseq=1, Sq=128, Sk=128)
    assert np.abs(o[:128].float().cpu().numpy() - o_ref).max() <= 1e-2


def test_rows_sum_to_one_and_constant_v():
    B, H, S, D = 2, 2, 640, 128
    q, k = _rand((B * S, H, D), torch.bfloat16, 31), _rand((B * S, H, D), torch.bfloat16, 32)
    for causal in (False, True):
        o, _ = _run(q, k, torch.ones_like(q), causal=causal, batch=B)
        assert (o.float() - 1).abs().max().item() <= 1e-2
        c = _rand((1, H, D), torch.bfloat16, 33)
        o, _ = _run(q, k, c.expand(B * S, H, D).contiguous(), causal=causal, batch=B)
        assert (o.float() - c.float()).abs().max().item() <= 1e-2


def test_causal_rows_ignore_future_bitwise():
    B, H, S, D = 1, 2, 700, 128
    q, k, v = (_rand((S, H, D), torch.bfloat16, 40 + i) for i in range(3))
    o1, l1 = _run(q, k, v, causal=True, batch=B)
    for cut in (0, 127, 300, 511):
        k2, v2 = k.clone(), v.clone()
        k2[cut + 1:] = _rand(k2[cut + 1:].shape, torch.bfloat16, 50 + cut, scale=4.0)
        v2[cut + 1:] = -v2[cut + 1:] + 1
        o2, l2 = _run(q, k2, v2, causal=True, batch=B)
        assert torch.equal(o1[:cut + 1], o2[:cut + 1]), cut
        assert torch.equal(l1[:, :, :cut + 1], l2[:, :, :cut + 1]), cut


def test_key_permutation_and_linearity():
    B, H, S, D = 1, 2, 384, 64
    q, k, v, v2 = (_rand((S, H, D), torch.float16, 60 + i) for i in range(4))
    o, lse = _run(q, k, v, causal=False, batch=B)
    perm = torch.randperm(S, generator=torch.Generator().manual_seed(0)).cuda()
    op, lp = _run(q, k[perm].contiguous(), v[perm].contiguous(), causal=False, batch=B)
    assert (o.float() - op.float()).abs().max().item() <= 2e-3
    assert (lse - lp).abs().max().item() <= 1e-3
    o2, _ = _run(q, k, v2, causal=False, batch=B)
    vs = (0.5 * v.float() + 0.25 * v2.float()).to(torch.float16)
    os_, _ = _run(q, k, vs, causal=False, batch=B)
    assert (os_.float() - (0.5 * o.float() + 0.25 * o2.float())).abs().max().item() <= 2e-3


def test_deterministic():
    q, k, v = (_rand((2 * 1000, 4, 128), torch.bfloat16, 70 + i) for i in range(3))
    a = _run(q, k, v, causal=True, batch=2)
    b = _run(q, k, v, causal=True, batch=2)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def _sampled(name, n_rows=2048):
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w, device="cuda")
    q, k, v = inp["q"], inp["k"], inp["v"]
    scale = w.D ** -0.5
    if w.varlen:
        cu = inp["cu_seqlens_q"]
        o, lse = _run(q, k, v, causal=w.causal, scale=scale, cu_seqlens_q=cu, cu_seqlens_k=cu,
                      max_seqlen_q=inp["max_seqlen"], max_seqlen_k=inp["max_seqlen"])
        kw = dict(cu_seqlens_q=cu.cpu(), cu_seqlens_k=cu.cpu())
        starts = cu.cpu().tolist()
    else:
        o, lse = _run(q, k, v, causal=w.causal, scale=scale, batch=w.B)
        kw = dict(Sq=w.Sq, Sk=w.Sk)
        starts = [b * w.Sq for b in range(w.B + 1)]
    rows = workloads.sample_rows(w, inp, n_rows)
    o_ref, lse_ref = orc.attention_rows(q, k, v, rows, scale=scale, causal=w.causal, nseq=w.B, **kw)
    idx_tok = torch.tensor([starts[b] + i for b, h, i in rows], device="cuda")
    idx_h = torch.tensor([h for b, h, i in rows], device="cuda")
    o_s = o[idx_tok, idx_h].float().cpu().numpy()
    if w.varlen:
        l_s = lse[idx_h, idx_tok].cpu().numpy()
    else:
        l_s = lse[torch.tensor([b for b, h, i in rows]), torch.tensor([h for b, h, i in rows]),
                  torch.tensor([i for b, h, i in rows])].cpu().numpy()
    return _check(torch.from_numpy(o_s), torch.from_numpy(l_s), o_ref, lse_ref, torch.bfloat16, name)


@pytest.mark.parametrize("name", ["c2", "c3a", "c3b", "c4"])
def test_full_size_sampled_rows(name):
    """The full-size workloads, launched exactly as the benchmark launches them,
    compared on a deterministic sample of >= 2048 rows (always rows 0, 127,
    128, 255, 256 and the last of every (sequence, head))."""
    _sampled(name)
