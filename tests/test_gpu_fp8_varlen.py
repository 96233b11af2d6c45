"""GPU parity of the variable-length FP8 path (fa_varlen_blocks,
fa_fp8_prep_varlen, fa_fwd_fp8_varlen) through the C ABI.

Same bars as the fixed-length FP8 tests (``tests/test_gpu_fp8.py``): per
sequence and head, codes and scales bit for bit against the FP8 oracle
(``oracle/fp8.py``, decisions in fp32); attention element by element within
twice the bounds of ``tests/fp8_bound.py`` and |LSE - LSE_ref| <= 1e-3. Where
the varlen path and the fixed-length path see the same problem, they must
agree bit for bit.
"""
import numpy as np
import pytest
import torch

from exact_attention_forward_tiled_gb300 import api
from exact_attention_forward_tiled_gb300 import build as fa_build
from oracle import fp8 as F
from tests import fp8_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    fa_build.build()
    api.lib()


def _rand(shape, seed, scale=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * scale).to(torch.bfloat16)


def _sigma(D, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randint(0, 2, (D,), generator=g, device="cuda", dtype=torch.int32) * 2 - 1).to(torch.int8)


def _cu(lengths):
    return torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device="cuda")


def _blocks(lengths):
    return np.concatenate([[0], np.cumsum([(n + 127) // 128 for n in lengths])]).astype(np.int64)


def _seq_head(prep, name, lens, b, h):
    """Codes [L_b, D] and scales [ceil(L_b / 128)] of sequence b, head h."""
    start = int(np.sum(lens[:b]))
    cb = _blocks(lens)
    codes = prep[name + "8"][start:start + lens[b], h, :].cpu().numpy()
    scales = prep[name + "_scale"][cb[b]:cb[b + 1], h].cpu().numpy()
    return codes, scales


def _check_seqs(prep, o, lse, lq, lk, H, scale, causal):
    """Every (sequence, head) with queries: element-wise against the oracle."""
    starts = np.concatenate([[0], np.cumsum(lq)])
    for b in range(len(lq)):
        if lq[b] == 0:
            continue
        for h in range(H):
            q8, qs = _seq_head(prep, "q", lq, b, h)
            k8, ks = _seq_head(prep, "k", lk, b, h)
            v8, vs = _seq_head(prep, "v", lk, b, h)
            og = o[starts[b]:starts[b + 1], h, :].float().cpu().numpy()
            lg = lse[h, starts[b]:starts[b + 1]].cpu().numpy()
            if lk[b] == 0:
                assert np.all(og == 0) and np.all(np.isneginf(lg))
                continue
            fp8_bound.check_attention(og, lg, q8, qs, k8, ks, v8, vs, np.arange(lq[b]), lq[b], scale=scale,
                                      causal=causal)


LQ = [1, 300, 128, 0, 257, 40]
LK = [129, 5, 400, 64, 0, 40]


@pytest.mark.parametrize("D", [64, 128, 256])
def test_varlen_blocks_and_prep_parity(D):
    """Block offsets match the host prefix sums; every sequence's blocks
    (counted from its own first token, short last block) match the oracle bit
    for bit."""
    H = 3
    q = _rand((sum(LQ), H, D), 1, 2.0)
    k = _rand((sum(LK), H, D), 2)
    v = _rand((sum(LK), H, D), 3, 0.5)
    v[130, 2, 9] = 50.0
    sigma = _sigma(D, 4)
    cq, ck = _cu(LQ), _cu(LK)
    prep = api.fp8_prepare_varlen(q, k, v, sigma, cu_seqlens_q=cq, cu_seqlens_k=ck, max_seqlen_q=max(LQ),
                                  max_seqlen_k=max(LK))
    api.fa_get_device_status()
    assert np.array_equal(prep["cu_blocks_q"].cpu().numpy(), _blocks(LQ))
    assert np.array_equal(prep["cu_blocks_k"].cpu().numpy(), _blocks(LK))
    sg = sigma.cpu().numpy()
    for name, x, lens, rot in (("q", q, LQ, sg), ("k", k, LK, sg), ("v", v, LK, None)):
        start = 0
        for b, n in enumerate(lens):
            for h in range(H):
                ref_codes, ref_s = F.prepare(x[start:start + n, h, :].cpu(), rot)
                codes, scales = _seq_head(prep, name, lens, b, h)
                assert np.array_equal(scales, ref_s), (name, b, h)
                assert np.array_equal(codes, ref_codes), (name, b, h)
            start += n


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_varlen_attention_elementwise(D, causal):
    H = 2
    q = _rand((sum(LQ), H, D), 10)
    k = _rand((sum(LK), H, D), 11)
    v = _rand((sum(LK), H, D), 12)
    cq, ck = _cu(LQ), _cu(LK)
    prep = api.fp8_prepare_varlen(q, k, v, _sigma(D, 13), cu_seqlens_q=cq, cu_seqlens_k=ck,
                                  max_seqlen_q=max(LQ), max_seqlen_k=max(LK))
    o, lse = api.fp8_attention_forward(prep, causal=causal)
    api.fa_get_device_status()
    _check_seqs(prep, o, lse, LQ, LK, H, D ** -0.5, causal)
    # rows with no visible key (the sequence with Lk = 0): O = 0
    s = sum(LQ[:4])
    assert np.all(o[s:s + LQ[4]].float().cpu().numpy() == 0)


def test_fp8_varlen_equals_fixed_length_bitwise():
    """Equal lengths: the varlen path and fa_fp8_prep + fa_fwd_fp8 give the
    same codes, the same scales (transposed layout) and the same O and LSE."""
    B, H, S, D = 3, 2, 300, 128
    q, k, v = (_rand((B * S, H, D), 20 + i) for i in range(3))
    sigma = _sigma(D, 23)
    fixed = api.fp8_prepare(q, k, v, sigma, batch=B)
    o1, lse1 = api.fp8_attention_forward(fixed, causal=True)
    cu = _cu([S] * B)
    var = api.fp8_prepare_varlen(q, k, v, sigma, cu_seqlens_q=cu, cu_seqlens_k=cu, max_seqlen_q=S,
                                 max_seqlen_k=S)
    o2, lse2 = api.fp8_attention_forward(var, causal=True)
    api.fa_get_device_status()
    nb = (S + 127) // 128
    for n in ("q", "k", "v"):
        assert torch.equal(fixed[n + "8"], var[n + "8"])
        fs = fixed[n + "_scale"]                               # [B, H, nb]
        vs = var[n + "_scale"][:B * nb].reshape(B, nb, H)      # [B*nb, H]
        assert torch.equal(fs, vs.permute(0, 2, 1))
    assert torch.equal(o1, o2)
    assert torch.equal(lse1.permute(1, 0, 2).reshape(H, B * S), lse2)


def test_fp8_varlen_kv_prepared_once_and_reused():
    """K/V prepared alone (no Q) and Q prepared alone give what one call on
    all three gives; the K/V preparation then serves a second Q."""
    H, D = 2, 128
    lq, lk = [70, 200, 1], [500, 129, 3000]
    q = _rand((sum(lq), H, D), 30)
    k = _rand((sum(lk), H, D), 31)
    v = _rand((sum(lk), H, D), 32)
    sigma = _sigma(D, 33)
    cq, ck = _cu(lq), _cu(lk)
    both = api.fp8_prepare_varlen(q, k, v, sigma, cu_seqlens_q=cq, cu_seqlens_k=ck, max_seqlen_q=max(lq),
                                  max_seqlen_k=max(lk))
    o1, lse1 = api.fp8_attention_forward(both, causal=True)
    kv = api.fp8_prepare_varlen(None, k, v, sigma, cu_seqlens_q=None, cu_seqlens_k=ck, max_seqlen_q=0,
                                max_seqlen_k=max(lk))
    qq = api.fp8_prepare_varlen(q, None, None, sigma, cu_seqlens_q=cq, cu_seqlens_k=None, max_seqlen_q=max(lq),
                                max_seqlen_k=0)
    o2, lse2 = api.fp8_attention_forward({**kv, **qq}, causal=True)
    api.fa_get_device_status()
    assert torch.equal(o1, o2) and torch.equal(lse1, lse2)
    # a second query batch against the same prepared cache
    q2 = _rand((sum(lq), H, D), 34)
    qq2 = api.fp8_prepare_varlen(q2, None, None, sigma, cu_seqlens_q=cq, cu_seqlens_k=None,
                                 max_seqlen_q=max(lq), max_seqlen_k=0)
    o3, lse3 = api.fp8_attention_forward({**kv, **qq2}, causal=True)
    api.fa_get_device_status()
    _check_seqs({**kv, **qq2}, o3, lse3, lq, lk, H, D ** -0.5, True)
    # causal rows of sequence 1 (Lq > Lk) that see no key
    assert not torch.isfinite(lse3).all()


def test_fp8_varlen_bad_block_offsets_are_reported():
    """Block offsets that do not match the lengths are refused by the kernels'
    own checks: FA_ERR_DEVICE_SEQLENS, and the other sequences still right."""
    H, D = 2, 128
    lens = [300, 200]
    q, k, v = (_rand((sum(lens), H, D), 40 + i) for i in range(3))
    cu = _cu(lens)
    prep = api.fp8_prepare_varlen(q, k, v, _sigma(D, 43), cu_seqlens_q=cu, cu_seqlens_k=cu, max_seqlen_q=300,
                                  max_seqlen_k=300)
    api.fa_get_device_status()
    o_ok, _ = api.fp8_attention_forward(prep)
    api.fa_get_device_status()
    bad = dict(prep)
    # sequence 0 has 3 key blocks, not 2; sequence 1 keeps its true offsets 3..5
    bad["cu_blocks_k"] = torch.tensor([1, 3, 5], dtype=torch.int32, device="cuda")
    o = torch.zeros_like(o_ok)
    api.fp8_attention_forward(bad, out=o)
    st, raw = api.fa_get_device_status(check=False)
    assert st == -6, (st, raw)
    assert torch.equal(o[300:], o_ok[300:])
    assert int(o[:300].abs().sum().item()) == 0


@pytest.mark.parametrize("seed", range(12))
def test_fp8_varlen_random_shapes(seed):
    """Seeded draws of head size, causal mask, softmax scale (0.5 to 2 times
    1/sqrt(D)), heads and per-sequence query / key lengths (empty ones
    included): codes and scales bit for bit, attention element by element."""
    r = np.random.default_rng(500 + seed)
    D = int(r.choice([64, 128, 256]))
    causal = bool(r.integers(2))
    H = int(r.integers(1, 4))
    n = int(r.integers(1, 6))
    lq = [int(x) if r.random() > 0.15 else 0 for x in r.integers(1, 700, size=n)]
    lk = [int(x) if r.random() > 0.15 else 0 for x in r.integers(1, 700, size=n)]
    if sum(lq) == 0 or sum(lk) == 0:
        lq[0], lk[0] = 77, 130
    scale = float(r.uniform(0.5, 2.0)) * D ** -0.5
    q = _rand((sum(lq), H, D), 600 + seed)
    k = _rand((sum(lk), H, D), 700 + seed)
    v = _rand((sum(lk), H, D), 800 + seed)
    sigma = _sigma(D, 900 + seed)
    cq, ck = _cu(lq), _cu(lk)
    prep = api.fp8_prepare_varlen(q, k, v, sigma, cu_seqlens_q=cq, cu_seqlens_k=ck, max_seqlen_q=max(lq),
                                  max_seqlen_k=max(lk))
    o, lse = api.fp8_attention_forward(prep, causal=causal, scale=scale)
    api.fa_get_device_status()
    sg = sigma.cpu().numpy()
    for name, x, lens, rot in (("q", q, lq, sg), ("k", k, lk, sg), ("v", v, lk, None)):
        start = 0
        for b, m in enumerate(lens):
            for h in range(H):
                ref_codes, ref_s = F.prepare(x[start:start + m, h, :].cpu(), rot)
                codes, scales = _seq_head(prep, name, lens, b, h)
                assert np.array_equal(scales, ref_s) and np.array_equal(codes, ref_codes), (name, b, h)
            start += m
    _check_seqs(prep, o, lse, lq, lk, H, scale, causal)
