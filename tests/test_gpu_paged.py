"""GPU parity of the paged-KV forward (fa_fwd_paged) through the C ABI.

Keys and values live in a cache of shuffled pages named by a block table
("Flash Attention 3 principles (guijiagi)" section 5.3). Paged attention is
attention over each sequence's keys in order, so the expected values are the
fp64 oracle on the keys gathered back into contiguous sequences (the gather
is plain indexing in the test); the bars are those of fa_fwd (max |dO| <= 1e-2
bf16, 2e-3 fp16, |dLSE| <= 1e-3). Without key ranges the paged path must also
equal fa_fwd's varlen path on the gathered tensors bit for bit: the kernel
sees the same tiles, only fetched from other rows.
"""
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


def _paged_problem(lens, Sq, H, D, page_size, dtype, seed, spare_pages=3):
    """Contiguous K/V per sequence, the same keys in a shuffled page cache,
    and the block table. Rows of a last page past the sequence hold finite
    noise; table entries past a sequence's pages hold an invalid index (never
    read)."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    B = len(lens)
    q = torch.randn((B * Sq, H, D), generator=g, device="cuda").to(dtype)
    k = torch.randn((sum(lens), H, D), generator=g, device="cuda").to(dtype)
    v = torch.randn((sum(lens), H, D), generator=g, device="cuda").to(dtype)
    pages_per = [(L + page_size - 1) // page_size for L in lens]
    max_pages = max(max(pages_per), 1)
    num_pages = sum(pages_per) + spare_pages
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(seed)).tolist()
    kc = torch.randn((num_pages, page_size, H, D), generator=g, device="cuda").to(dtype)
    vc = torch.randn((num_pages, page_size, H, D), generator=g, device="cuda").to(dtype)
    table = torch.full((B, max_pages), 10 ** 7, dtype=torch.int32)
    nxt, start = 0, 0
    for b, L in enumerate(lens):
        for j in range(pages_per[b]):
            pg = perm[nxt]
            nxt += 1
            table[b, j] = pg
            n = min(page_size, L - j * page_size)
            kc[pg, :n] = k[start + j * page_size:start + j * page_size + n]
            vc[pg, :n] = v[start + j * page_size:start + j * page_size + n]
        start += L
    seqlens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    return q, k, v, kc, vc, table.cuda(), seqlens


def _oracle(q, k, v, lens, Sq, scale, causal):
    B = len(lens)
    cq = np.arange(B + 1) * Sq
    ck = np.concatenate([[0], np.cumsum(lens)])
    o, lse = orc.attention(q.cpu(), k.cpu(), v.cpu(), scale=scale, causal=causal, nseq=B, cu_seqlens_q=cq,
                           cu_seqlens_k=ck)
    H = q.shape[1]
    return o, lse.reshape(H, B, Sq).transpose(1, 0, 2)   # -> [B, H, Sq]


def _check_vs_oracle(o, lse, o_ref, lse_ref, dtype):
    err = np.abs(o.float().cpu().numpy() - o_ref).max()
    assert err <= TOL_O[dtype], err
    l = lse.cpu().numpy()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(l), fin)
    if fin.any():
        assert np.abs(l[fin] - lse_ref[fin]).max() <= 1e-3


@pytest.mark.parametrize("page_size", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_paged_matches_oracle_and_varlen(page_size, D, causal):
    lens, Sq, H = [1, 300, 128, 0, 517, 64], 70, 2
    dtype = torch.float16 if D == 64 else torch.bfloat16
    q, k, v, kc, vc, table, seqlens = _paged_problem(lens, Sq, H, D, page_size, dtype, seed=page_size + D + causal)
    o, lse = api.attention_forward_paged(q, kc, vc, table, seqlens, causal=causal)
    api.fa_get_device_status()
    o_ref, lse_ref = _oracle(q, k, v, lens, Sq, D ** -0.5, causal)
    _check_vs_oracle(o, lse, o_ref, lse_ref, dtype)
    # the contiguous varlen path on the gathered keys: bit for bit
    cq = torch.arange(len(lens) + 1, dtype=torch.int32, device="cuda") * Sq
    ck = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    o2, lse2 = api.attention_forward(q, k, v, causal=causal, cu_seqlens_q=cq, cu_seqlens_k=ck, max_seqlen_q=Sq,
                                     max_seqlen_k=max(lens))
    api.fa_get_device_status()
    assert torch.equal(o, o2)
    assert torch.equal(lse, lse2.reshape(H, len(lens), Sq).permute(1, 0, 2))


@pytest.mark.parametrize("splits", [0, 3])
def test_paged_decode_with_key_ranges(splits):
    """Decode shape: one query per sequence against long paged contexts,
    cut into key ranges and merged."""
    lens, Sq, H, D = [4000, 1, 2500, 8191, 129], 1, 4, 128
    q, k, v, kc, vc, table, seqlens = _paged_problem(lens, Sq, H, D, 16, torch.bfloat16, seed=40 + splits)
    o, lse = api.attention_forward_paged(q, kc, vc, table, seqlens, causal=True, num_splits=splits)
    api.fa_get_device_status()
    o_ref, lse_ref = _oracle(q, k, v, lens, Sq, D ** -0.5, True)
    _check_vs_oracle(o, lse, o_ref, lse_ref, torch.bfloat16)


def test_paged_bad_page_entry_is_reported():
    """A block-table entry outside the cache is never dereferenced: its keys
    read as zeros, the status word says so, the other sequences are right."""
    lens, Sq, H, D = [300, 200], 64, 2, 128
    q, k, v, kc, vc, table, seqlens = _paged_problem(lens, Sq, H, D, 64, torch.bfloat16, seed=7)
    table[0, 2] = kc.shape[0] + 5
    o, lse = api.attention_forward_paged(q, kc, vc, table, seqlens)
    st, raw = api.fa_get_device_status(check=False)
    assert st == -6, (st, raw)
    o_ref, lse_ref = _oracle(q, k, v, lens, Sq, D ** -0.5, False)
    assert np.abs(o[Sq:].float().cpu().numpy() - o_ref[Sq:]).max() <= 1e-2
    # and a length beyond the table is refused for that sequence only
    seqlens[1] = table.shape[1] * 64 + 1
    api.attention_forward_paged(q, kc, vc, table, seqlens)
    st, raw = api.fa_get_device_status(check=False)
    assert st == -6


def test_paged_host_checks():
    lens, Sq, H, D = [100], 8, 1, 64
    q, k, v, kc, vc, table, seqlens = _paged_problem(lens, Sq, H, D, 32, torch.float16, seed=9)
    o = torch.empty_like(q)
    lse = torch.empty((1, H, Sq), device="cuda")
    for ps in (8, 48, 100):
        st = api.fa_fwd_paged(q, kc, vc, table, seqlens, o, lse, 1, H, Sq, D, kc.shape[0], ps, table.shape[1],
                              0.125, 0, check=False)
        assert st == -1, ps
    st = api.fa_fwd_paged(q, kc, vc, None, seqlens, o, lse, 1, H, Sq, D, kc.shape[0], 32, table.shape[1], 0.125, 0,
                          check=False)
    assert st == -1


@pytest.mark.parametrize("causal", [False, True])
def test_paged_packed_queries(causal):
    """Chunked prefill: a different number of new queries per sequence
    (packed by cu_seqlens_q) against paged contexts; equal, bit for bit, to
    the contiguous varlen path on the gathered keys."""
    H, D, ps = 2, 128, 16
    lq, lk = [5, 130, 1, 0, 64], [300, 200, 1, 50, 1000]
    _, k, v, kc, vc, table, seqlens = _paged_problem(lk, 1, H, D, ps, torch.bfloat16, seed=60 + causal)
    g = torch.Generator(device="cuda").manual_seed(61)
    q = torch.randn((sum(lq), H, D), generator=g, device="cuda").to(torch.bfloat16)
    cq = torch.tensor(np.concatenate([[0], np.cumsum(lq)]), dtype=torch.int32, device="cuda")
    ck = torch.tensor(np.concatenate([[0], np.cumsum(lk)]), dtype=torch.int32, device="cuda")
    o, lse = api.attention_forward_paged(q, kc, vc, table, seqlens, causal=causal, cu_seqlens_q=cq,
                                         max_seqlen_q=max(lq))
    api.fa_get_device_status()
    o_ref, lse_ref = orc.attention(q.cpu(), k.cpu(), v.cpu(), scale=D ** -0.5, causal=causal, nseq=len(lq),
                                   cu_seqlens_q=cq.cpu().numpy(), cu_seqlens_k=ck.cpu().numpy())
    _check_vs_oracle(o, lse, o_ref, lse_ref, torch.bfloat16)
    o2, lse2 = api.attention_forward(q, k, v, causal=causal, cu_seqlens_q=cq, cu_seqlens_k=ck,
                                     max_seqlen_q=max(lq), max_seqlen_k=max(lk))
    api.fa_get_device_status()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    # packed queries take one launch: key ranges are refused
    st = api.fa_fwd_paged(q, kc, vc, table, seqlens, o, lse, len(lq), H, max(lq), D, kc.shape[0], ps,
                          table.shape[1], D ** -0.5, causal, num_splits=2, cu_seqlens_q=cq, total_q=q.shape[0],
                          check=False)
    assert st == -2


def test_paged_key_ranges_with_several_queries():
    """Key ranges with more than one query row per sequence (causal): the
    merge of the ranges equals the oracle."""
    lens, Sq, H, D = [900, 1500, 70], 70, 2, 128
    q, k, v, kc, vc, table, seqlens = _paged_problem(lens, Sq, H, D, 32, torch.bfloat16, seed=70)
    o, lse = api.attention_forward_paged(q, kc, vc, table, seqlens, causal=True, num_splits=3)
    api.fa_get_device_status()
    o_ref, lse_ref = _oracle(q, k, v, lens, Sq, D ** -0.5, True)
    _check_vs_oracle(o, lse, o_ref, lse_ref, torch.bfloat16)


@pytest.mark.parametrize("seed", range(10))
def test_paged_random_shapes(seed):
    """Seeded draws of page size, head size, mask, query length and per-
    sequence key lengths (empty ones included): the oracle's bars, and bit
    equality with the contiguous varlen path on the gathered keys."""
    r = np.random.default_rng(9000 + seed)
    page_size = int(r.choice([16, 32, 64, 128, 256]))
    D = int(r.choice([64, 128, 256]))
    causal = bool(r.integers(2))
    H = int(r.integers(1, 3))
    n = int(r.integers(1, 6))
    lens = [int(x) if r.random() > 0.15 else 0 for x in r.integers(1, 900, size=n)]
    if sum(lens) == 0:
        lens[0] = 333
    Sq = int(r.integers(1, 200))
    dtype = [torch.float16, torch.bfloat16][r.integers(2)]
    q, k, v, kc, vc, table, seqlens = _paged_problem(lens, Sq, H, D, page_size, dtype, seed=9100 + seed)
    o, lse = api.attention_forward_paged(q, kc, vc, table, seqlens, causal=causal)
    api.fa_get_device_status()
    o_ref, lse_ref = _oracle(q, k, v, lens, Sq, D ** -0.5, causal)
    # the 16-bit bar plus one unit of the output type's rounding times |O_ref|
    # (rows that see one or two keys have |O| near max |V|)
    rel = 2.0 ** -11 if dtype == torch.float16 else 2.0 ** -8
    err = np.abs(o.float().cpu().numpy() - o_ref)
    assert (err / (TOL_O[dtype] + rel * np.abs(o_ref))).max() <= 1.0
    l = lse.cpu().numpy()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(l), fin)
    if fin.any():
        assert np.abs(l[fin] - lse_ref[fin]).max() <= 1e-3
    cq = torch.arange(len(lens) + 1, dtype=torch.int32, device="cuda") * Sq
    ck = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    o2, lse2 = api.attention_forward(q, k, v, causal=causal, cu_seqlens_q=cq, cu_seqlens_k=ck, max_seqlen_q=Sq,
                                     max_seqlen_k=max(lens))
    api.fa_get_device_status()
    assert torch.equal(o, o2)
    assert torch.equal(lse, lse2.reshape(H, len(lens), Sq).permute(1, 0, 2))
