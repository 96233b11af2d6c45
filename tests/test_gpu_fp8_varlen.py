"""GPU parity of the variable-length FP8 path (fa_varlen_blocks,
fa_fp8_prep_varlen, fa_fwd_fp8_varlen) through the C ABI.

Same bars as the fixed-length FP8 tests: per sequence and head, scales within
fp32 rounding of the oracle's and e4m3 codes at most one code apart; attention
against the fp64 oracle on the dequantised inputs with a normalised RMSE of
5 % and |LSE - LSE_ref| <= 1e-3. Where the varlen path and the fixed-length
path see the same problem, they must agree bit for bit.
"""
import numpy as np
import pytest
import torch

from exact_attention_forward_tiled_gb300 import api
from exact_attention_forward_tiled_gb300 import build as fa_build
from oracle import oracle as orc

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


def _signed_index(codes):
    c = codes.astype(np.int64)
    return np.where(c & 0x80, -(c & 0x7F), c & 0x7F)


def _oracle_prep(x, sigma):
    x = orc._f64(x)
    if sigma is not None:
        x = x @ orc.rotation(sigma.cpu().numpy().astype(np.float64))
    s = orc.block_scales(x)
    codes = np.concatenate([orc.e4m3_encode(x[b * 128:(b + 1) * 128] / s[b]) for b in range(len(s))]) \
        if len(s) else np.zeros((0, x.shape[1]), np.uint8)
    return codes, s


def _dequant(codes, scales, lengths):
    """codes [total, H, D] e4m3, scales [n_blocks, H] -> fp64 values."""
    val = orc.e4m3_decode(codes.cpu().numpy())
    sc = scales.cpu().numpy()
    cb = _blocks(lengths)
    starts = np.concatenate([[0], np.cumsum(lengths)])
    out = np.empty_like(val)
    for b, n in enumerate(lengths):
        for blk in range((n + 127) // 128):
            r0, r1 = starts[b] + blk * 128, starts[b] + min(blk * 128 + 128, n)
            out[r0:r1] = val[r0:r1] * sc[cb[b] + blk][None, :, None]
    return out


LQ = [1, 300, 128, 0, 257, 40]
LK = [129, 5, 400, 64, 0, 40]


@pytest.mark.parametrize("D", [64, 128, 256])
def test_varlen_blocks_and_prep_parity(D):
    """Block offsets match the host prefix sums; every sequence's blocks
    (counted from its own first token, short last block) match the oracle."""
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
    for name, x, lens, sg in (("q", q, LQ, sigma), ("k", k, LK, sigma), ("v", v, LK, None)):
        codes = prep[name + "8"].cpu().numpy()
        scales = prep[name + "_scale"].cpu().numpy()
        cb = _blocks(lens)
        start = 0
        for b, n in enumerate(lens):
            for h in range(H):
                ref_codes, ref_s = _oracle_prep(x[start:start + n, h, :].cpu(), sg)
                np.testing.assert_allclose(scales[cb[b]:cb[b + 1], h], ref_s, rtol=2e-6, err_msg=name)
                d = np.abs(_signed_index(codes[start:start + n, h, :]) - _signed_index(ref_codes))
                if n:
                    assert d.max() <= 1, (name, b, h)
            start += n


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_varlen_attention_matches_dequantized(D, causal):
    H = 2
    q = _rand((sum(LQ), H, D), 10)
    k = _rand((sum(LK), H, D), 11)
    v = _rand((sum(LK), H, D), 12)
    cq, ck = _cu(LQ), _cu(LK)
    prep = api.fp8_prepare_varlen(q, k, v, _sigma(D, 13), cu_seqlens_q=cq, cu_seqlens_k=ck,
                                  max_seqlen_q=max(LQ), max_seqlen_k=max(LK))
    o, lse = api.fp8_attention_forward(prep, causal=causal)
    api.fa_get_device_status()
    qd = _dequant(prep["q8"], prep["q_scale"], LQ)
    kd = _dequant(prep["k8"], prep["k_scale"], LK)
    vd = _dequant(prep["v8"], prep["v_scale"], LK)
    o_ref, lse_ref = orc.attention(qd, kd, vd, scale=D ** -0.5, causal=causal, nseq=len(LQ),
                                   cu_seqlens_q=cq.cpu().numpy(), cu_seqlens_k=ck.cpu().numpy())
    o = o.float().cpu().numpy()
    nrmse = np.linalg.norm(o - o_ref) / np.linalg.norm(o_ref)
    assert nrmse <= 0.05, nrmse
    l = lse.cpu().numpy()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(l), fin)
    assert np.abs(l[fin] - lse_ref[fin]).max() <= 1e-3
    # rows with no visible key (the sequence with Lk = 0): O = 0
    s = sum(LQ[:4])
    assert np.all(o[s:s + LQ[4]] == 0)


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
    qd = _dequant(qq2["q8"], qq2["q_scale"], lq)
    kd = _dequant(kv["k8"], kv["k_scale"], lk)
    vd = _dequant(kv["v8"], kv["v_scale"], lk)
    o_ref, lse_ref = orc.attention(qd, kd, vd, scale=D ** -0.5, causal=True, nseq=len(lq),
                                   cu_seqlens_q=cq.cpu().numpy(), cu_seqlens_k=ck.cpu().numpy())
    o3 = o3.float().cpu().numpy()
    assert np.linalg.norm(o3 - o_ref) / np.linalg.norm(o_ref) <= 0.05
    l3 = lse3.cpu().numpy()
    fin = np.isfinite(lse_ref)   # causal rows of sequence 1 (Lq > Lk) see no key
    assert np.array_equal(np.isfinite(l3), fin) and not fin.all()
    assert np.abs(l3[fin] - lse_ref[fin]).max() <= 1e-3


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
