"""Randomised GPU parity of the 16-bit forward against the fp64 oracle, every
element: seeded draws of input type, head size, causal mask, softmax scale
(0.5 to 2.5 times 1/sqrt(D)) and shape. Fixed-length batches take random
Sq != Sk; varlen batches take random query and key lengths per sequence,
including empty ones and lengths that straddle the 128-row tiles.

Bars: max |LSE - LSE_ref| <= 1e-3, and |O - O_ref| <= 2e-3 (fp16) or 1e-2
(bf16) plus one unit of the output type's relative rounding times |O_ref|
(2^-11 fp16, 2^-8 bf16). The absolute bars hold for the averaged outputs of
many keys (|O| well below 1). Causal rows with Sq > Sk see one or two keys,
so |O| approaches max |V| (about 4 for N(0, 1) V). An O of 4 in bf16 is
rounded to a spacing of 2^-5 and P to 2^-9 of its size, so no bf16
attention can hold 1e-2 absolute there."""
import numpy as np
import pytest
import torch

from exact_attention_forward_tiled_gb300 import api
from exact_attention_forward_tiled_gb300 import build as fa_build
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

TOL_O = {torch.float16: 2e-3, torch.bfloat16: 1e-2}
REL_O = {torch.float16: 2.0 ** -11, torch.bfloat16: 2.0 ** -8}
TOL_LSE = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    fa_build.build()
    api.lib()


def _case(seed):
    r = np.random.default_rng(seed)
    return dict(dtype=[torch.float16, torch.bfloat16][r.integers(2)], D=int(r.choice([64, 128, 256])),
                causal=bool(r.integers(2)), H=int(r.integers(1, 5)), scale_mul=float(r.uniform(0.5, 2.5)),
                rng=r)


def _inputs(T_q, T_k, H, D, dtype, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn((T_q, H, D), generator=g, device="cuda").to(dtype)
    k = torch.randn((T_k, H, D), generator=g, device="cuda").to(dtype)
    v = torch.randn((T_k, H, D), generator=g, device="cuda").to(dtype)
    return q, k, v


def _compare(o, lse, o_ref, lse_ref, dtype, what):
    api.fa_get_device_status()
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: -inf pattern of LSE differs"
    # worst ratio of the error to its bar, element by element
    bar = TOL_O[dtype] + REL_O[dtype] * np.abs(o_ref)
    ratio = (np.abs(o - o_ref) / bar).max() if o.size else 0.0
    err_l = np.abs(lse[fin] - lse_ref[fin]).max() if fin.any() else 0.0
    assert ratio <= 1.0, f"{what}: |dO| / bar = {ratio:.3f}"
    assert err_l <= TOL_LSE, f"{what}: max|dLSE| = {err_l:.3e}"


@pytest.mark.parametrize("seed", range(18))
def test_random_fixed_length(seed):
    c = _case(1000 + seed)
    r = c["rng"]
    B = int(r.integers(1, 4))
    Sq, Sk = (int(x) for x in r.integers(1, 700, size=2))
    D, H, dtype, causal = c["D"], c["H"], c["dtype"], c["causal"]
    scale = c["scale_mul"] * D ** -0.5
    q, k, v = _inputs(B * Sq, B * Sk, H, D, dtype, 2000 + seed)
    o, lse = api.attention_forward(q, k, v, causal=causal, scale=scale, batch=B)
    o_ref, lse_ref = orc.attention(q.cpu(), k.cpu(), v.cpu(), scale=scale, causal=causal, nseq=B, Sq=Sq, Sk=Sk)
    _compare(o, lse, o_ref, lse_ref, dtype, f"B{B} H{H} Sq{Sq} Sk{Sk} D{D} causal={causal} {dtype}")


@pytest.mark.parametrize("seed", range(18))
def test_random_varlen(seed):
    c = _case(3000 + seed)
    r = c["rng"]
    n = int(r.integers(1, 7))
    lq = [int(x) if r.random() > 0.15 else 0 for x in r.integers(1, 600, size=n)]
    lk = [int(x) if r.random() > 0.15 else 0 for x in r.integers(1, 600, size=n)]
    D, H, dtype, causal = c["D"], c["H"], c["dtype"], c["causal"]
    scale = c["scale_mul"] * D ** -0.5
    cq = torch.tensor([0] + list(np.cumsum(lq)), dtype=torch.int32, device="cuda")
    ck = torch.tensor([0] + list(np.cumsum(lk)), dtype=torch.int32, device="cuda")
    q, k, v = _inputs(int(cq[-1]), int(ck[-1]), H, D, dtype, 4000 + seed)
    o, lse = api.attention_forward(q, k, v, causal=causal, scale=scale, cu_seqlens_q=cq, cu_seqlens_k=ck,
                                   max_seqlen_q=max(lq), max_seqlen_k=max(lk))
    o_ref, lse_ref = orc.attention(q.cpu(), k.cpu(), v.cpu(), scale=scale, causal=causal, nseq=n,
                                   cu_seqlens_q=cq.cpu(), cu_seqlens_k=ck.cpu())
    _compare(o, lse, o_ref, lse_ref, dtype, f"varlen lq={lq} lk={lk} H{H} D{D} causal={causal} {dtype}")


@pytest.mark.parametrize("varlen", [False, True])
def test_no_key_rows_at_all(varlen):
    """Query rows but no key rows (Sk = 0, or every key length 0): every row
    gets O = 0 and LSE = -inf, and empty K, V tensors are accepted."""
    H, D, dtype = 2, 128, torch.bfloat16
    lq = [5, 300, 129]
    q, k, v = _inputs(sum(lq), 0, H, D, dtype, 77)
    if varlen:
        cq = torch.tensor([0] + list(np.cumsum(lq)), dtype=torch.int32, device="cuda")
        ck = torch.zeros(len(lq) + 1, dtype=torch.int32, device="cuda")
        o, lse = api.attention_forward(q, k, v, causal=False, scale=D ** -0.5, cu_seqlens_q=cq,
                                       cu_seqlens_k=ck, max_seqlen_q=max(lq), max_seqlen_k=0)
    else:
        q = q[:3 * 100]
        o, lse = api.attention_forward(q, k, v, causal=False, scale=D ** -0.5, batch=3)
    api.fa_get_device_status()
    assert torch.count_nonzero(o) == 0
    assert torch.isneginf(lse).all()
