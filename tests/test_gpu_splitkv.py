"""GPU parity of the split-KV forward (fa_fwd_splitkv) through the C ABI:
against the fp64 oracle (same bars as fa_fwd: max |O - O_ref| <= 2e-3 fp16,
<= 1e-2 bf16, |LSE - LSE_ref| <= 1e-3) and against fa_fwd itself."""
import numpy as np
import pytest
import torch

from exact_attention_forward_tiled_gb300 import api
from exact_attention_forward_tiled_gb300 import build as fa_build
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

TOL_O = {torch.float16: 2e-3, torch.bfloat16: 1e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    fa_build.build()
    api.lib()


def _rand(shape, dtype, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(shape, generator=g, device="cuda").to(dtype)


def _case(B, H, Sq, Sk, D, causal, num_splits, dtype, seed):
    q = _rand((B * Sq, H, D), dtype, seed)
    k = _rand((B * Sk, H, D), dtype, seed + 1)
    v = _rand((B * Sk, H, D), dtype, seed + 2)
    o, lse = api.attention_forward_splitkv(q, k, v, batch=B, causal=causal, num_splits=num_splits)
    api.fa_get_device_status()
    o_ref, lse_ref = orc.attention(q.cpu(), k.cpu(), v.cpu(), scale=D ** -0.5, causal=causal, nseq=B,
                                   Sq=Sq, Sk=Sk)
    err_o = np.abs(o.float().cpu().numpy() - o_ref).max()
    l = lse.cpu().numpy()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(l), fin)
    err_l = np.abs(l[fin] - lse_ref[fin]).max() if fin.any() else 0.0
    assert err_o <= TOL_O[dtype], err_o
    assert err_l <= 1e-3, err_l
    return q, k, v, o, lse


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Sq,Sk,splits", [(1, 1000, 0), (100, 4097, 3), (256, 2048, 0), (300, 300, 7),
                                          (130, 129, 2)])
def test_splitkv_matches_oracle(D, causal, Sq, Sk, splits):
    dtype = torch.float16 if D == 64 else torch.bfloat16
    _case(2, 3, Sq, Sk, D, causal, splits, dtype, seed=D + Sq + Sk + causal)


def test_splitkv_agrees_with_unsplit_forward():
    B, H, Sq, Sk, D = 1, 4, 256, 8192, 128
    q, k, v, o, lse = _case(B, H, Sq, Sk, D, False, 0, torch.bfloat16, seed=5)
    o1, lse1 = api.attention_forward(q, k, v, batch=B)
    api.fa_get_device_status()
    assert (o.float() - o1.float()).abs().max().item() <= 1e-2
    assert (lse - lse1).abs().max().item() <= 1e-3


def test_splitkv_single_split_equals_unsplit_bitwise_lse_range():
    """With one range the partial results are the whole rows; the merge only
    re-rounds O to bf16, so O matches fa_fwd exactly and LSE to fp32 rounding."""
    B, H, Sq, Sk, D = 2, 2, 200, 700, 128
    q, k, v = (_rand((B * s, H, D), torch.bfloat16, 30 + i) for i, s in enumerate((Sq, Sk, Sk)))
    o, lse = api.attention_forward_splitkv(q, k, v, batch=B, num_splits=1)
    o1, lse1 = api.attention_forward(q, k, v, batch=B)
    api.fa_get_device_status()
    assert torch.equal(o, o1)
    assert (lse - lse1).abs().max().item() <= 1e-5


def test_splitkv_workspace_too_small_is_rejected():
    B, H, Sq, Sk, D = 1, 2, 128, 1024, 64
    q, k, v = (_rand((B * s, H, D), torch.float16, 40 + i) for i, s in enumerate((Sq, Sk, Sk)))
    need = api.fa_fwd_splitkv_workspace_size(B, H, Sq, Sk, D, 4)
    assert need > 0
    ws = torch.empty(need - 4, dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Sq), device="cuda")
    st = api.fa_fwd_splitkv(q, k, v, o, lse, B, H, Sq, Sk, D, 0.125, 0, 4, ws, need - 4, check=False)
    assert st == -1


def test_splitkv_full_size_sampled_rows():
    """The split-KV workload (B=2 H=8 Sq=256 Sk=65536 D=128), launched as the
    benchmark launches it, on sampled rows."""
    from exact_attention_forward_tiled_gb300 import workloads
    w = workloads.WORKLOADS["f1"]
    inp = workloads.make_inputs(w, device="cuda")
    q, k, v = inp["q"], inp["k"], inp["v"]
    o, lse = api.attention_forward_splitkv(q, k, v, batch=w.B, num_splits=0)
    api.fa_get_device_status()
    rows = workloads.sample_rows(w, inp, 256)
    o_ref, lse_ref = orc.attention_rows(q, k, v, rows, scale=w.D ** -0.5, causal=False, nseq=w.B,
                                        Sq=w.Sq, Sk=w.Sk)
    tok = torch.tensor([b * w.Sq + i for b, h, i in rows], device="cuda")
    hh = torch.tensor([h for b, h, i in rows], device="cuda")
    bb = torch.tensor([b for b, h, i in rows], device="cuda")
    ii = torch.tensor([i for b, h, i in rows], device="cuda")
    assert np.abs(o[tok, hh].float().cpu().numpy() - o_ref).max() <= 1e-2
    assert np.abs(lse[bb, hh, ii].cpu().numpy() - lse_ref).max() <= 1e-3
