"""Seeded synthetic inputs for the attention forward workloads.

This module holds the shapes, seeds and random draws only; none of the
method's arithmetic. Both the CUDA path and the oracle consume what it makes.

The pages benchmark unspecified synthetic shapes ("Flash Attention 3
principles (guijiagi)" section 4.2 table: causal 4K/8K/16K and full 8K; the
FlashAttention-3 wiki's hdim-128/256 figures). The workloads below stand in
for them: Q, K, V i.i.d. N(0, 1) drawn in fp32 and cast to the input dtype.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str            # "fp16" | "bf16" | "fp8"  (fp8: bf16 inputs, e4m3 compute)
    B: int                # sequences (fixed length) or number of varlen sequences
    H: int
    Sq: int               # fixed: query length; varlen: max length
    Sk: int
    D: int
    causal: bool
    seed: int
    varlen: bool = False
    len_range: tuple = (128, 8192)   # varlen: inclusive uniform range of lengths
    outliers: bool = False           # fp8 outlier workload
    splitkv: bool = False            # run through the split-KV forward
    backward: bool = False           # forward + backward step (an upstream gradient dO is drawn too)
    page_size: int = 0               # > 0: K/V also laid out in a paged cache of this page size
    note: str = field(default="", compare=False)


WORKLOADS = {
    "c1": Workload("fp16_B1_H2_S256_D64", "fp16", 1, 2, 256, 256, 64, False, 0,
                   note="fp16 B=1 H=2 Sq=Sk=256 D=64 non-causal, scale 1/sqrt(D), seed 0"),
    "c2": Workload("bf16_B4_H16_S8192_D128", "bf16", 4, 16, 8192, 8192, 128, False, 1,
                   note="bf16 B=4 H=16 Sq=Sk=8192 D=128 non-causal"),
    "c3a": Workload("bf16_causal_B2_H16_S16384_D128", "bf16", 2, 16, 16384, 16384, 128, True, 2,
                    note="bf16 causal B=2 H=16 Sq=Sk=16384 D=128"),
    "c3b": Workload("bf16_causal_B1_H8_S16384_D256", "bf16", 1, 8, 16384, 16384, 256, True, 3,
                    note="bf16 causal B=1 H=8 Sq=Sk=16384 D=256"),
    "c4": Workload("bf16_varlen_causal_32seq_H32_D128", "bf16", 32, 32, 8192, 8192, 128, True, 4,
                   varlen=True, note="bf16 varlen causal, 32 sequences of U[128, 8192] tokens, H=32 D=128"),
    "c5": Workload("fp8_B4_H16_S8192_D128_outliers", "fp8", 4, 16, 8192, 8192, 128, False, 5,
                   outliers=True,
                   note="fp8 e4m3 B=4 H=16 Sq=Sk=8192 D=128 non-causal, block scales + Hadamard, "
                        "0.1% N(0,10^2) outliers in 4 fixed columns"),
    # split-KV: few query rows against a long key sequence, where B*H*ceil(Sq/256)
    # = 16 work tiles alone would leave most SMs idle
    "f1": Workload("bf16_splitkv_B2_H8_Sq256_Sk65536_D128", "bf16", 2, 8, 256, 65536, 128, False, 6,
                   splitkv=True, note="bf16 split-KV B=2 H=8 Sq=256 Sk=65536 D=128 non-causal"),
    # backward: the forward's shapes with an upstream gradient dO ~ N(0, 1)
    "b1": Workload("bf16_bwd_B4_H16_S8192_D128", "bf16", 4, 16, 8192, 8192, 128, False, 7, backward=True,
                   note="bf16 backward B=4 H=16 Sq=Sk=8192 D=128 non-causal"),
    "b2": Workload("bf16_bwd_causal_B2_H16_S16384_D128", "bf16", 2, 16, 16384, 16384, 128, True, 8,
                   backward=True, note="bf16 backward causal B=2 H=16 Sq=Sk=16384 D=128"),
    "b3": Workload("bf16_bwd_causal_B1_H8_S16384_D256", "bf16", 1, 8, 16384, 16384, 256, True, 11,
                   backward=True, note="bf16 backward causal B=1 H=8 Sq=Sk=16384 D=256 (the c3b shape)"),
    # paged K/V: Sq new queries per sequence at the end of an Sk-key context
    # whose keys sit in shuffled 16-key pages
    "p1": Workload("bf16_paged_prefill_B8_H16_Sq1024_Sk8192_D128_page16", "bf16", 8, 16, 1024, 8192, 128, True, 9,
                   page_size=16, note="bf16 paged, chunked prefill: B=8 H=16, 1024 new queries against 8192 "
                                      "cached keys (causal, bottom-right), pages of 16 keys, D=128"),
    "p2": Workload("bf16_paged_decode_B64_H16_Sq1_Sk8192_D128_page16", "bf16", 64, 16, 1, 8192, 128, True, 10,
                   page_size=16, note="bf16 paged decode: B=64 H=16, one query against 8192 cached keys, "
                                      "pages of 16 keys, D=128, automatic key ranges"),
}

TORCH_DTYPE = {"fp16": torch.float16, "bf16": torch.bfloat16, "fp8": torch.bfloat16}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def varlen_lengths(w: Workload, device="cpu") -> torch.Tensor:
    """Sequence lengths, i.i.d. uniform on ``len_range`` (inclusive), drawn
    first from the workload's seed on the CPU (so both machines agree)."""
    g = _gen(w.seed, "cpu")
    lo, hi = w.len_range
    return torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int64)


def cu_seqlens(lengths: torch.Tensor) -> torch.Tensor:
    """int32 prefix sums [0, L0, L0+L1, ...]."""
    out = torch.zeros(lengths.numel() + 1, dtype=torch.int64)
    out[1:] = torch.cumsum(lengths.to(torch.int64), 0)
    return out.to(torch.int32)


def make_inputs(w: Workload, device="cpu", seed: Optional[int] = None):
    """Q, K, V of the workload as ``[tokens, H, D]`` tensors on ``device``.

    Returns a dict with q, k, v, cu_seqlens_q/k (None unless varlen), the
    lengths and, for the FP8 workload, sigma (int8 +-1 of length D) and the
    outlier columns; for a backward workload also dO (drawn after V). Random numbers come from a ``torch.Generator`` on
    ``device`` seeded with the workload's seed.
    """
    seed = w.seed if seed is None else seed
    dt = TORCH_DTYPE[w.dtype]
    out = {"cu_seqlens_q": None, "cu_seqlens_k": None}
    if w.varlen:
        lens = varlen_lengths(replace(w, seed=seed))
        cu = cu_seqlens(lens)
        out["lengths"] = lens
        out["cu_seqlens_q"] = cu.to(device)
        out["cu_seqlens_k"] = cu.to(device)
        out["max_seqlen"] = int(lens.max())
        Tq = Tk = int(cu[-1])
    else:
        Tq, Tk = w.B * w.Sq, w.B * w.Sk
    g = _gen(seed, device)
    q = torch.randn((Tq, w.H, w.D), generator=g, device=device, dtype=torch.float32)
    k = torch.randn((Tk, w.H, w.D), generator=g, device=device, dtype=torch.float32)
    v = torch.randn((Tk, w.H, w.D), generator=g, device=device, dtype=torch.float32)
    if w.outliers:
        # 4 distinct feature columns shared by Q, K, V and every head; in each
        # tensor round(0.001 * numel) entries of those columns, chosen
        # uniformly without replacement, become N(0, 10^2) draws.
        cols = torch.randperm(w.D, generator=g, device=device)[:4]
        out["outlier_cols"] = cols.cpu()
        for t in (q, k, v):
            n_out = int(round(0.001 * t.numel()))
            cand = t.shape[0] * t.shape[1] * 4
            pick = torch.randperm(cand, generator=g, device=device)[:n_out]
            col = cols[pick % 4]
            rest = pick // 4
            head = rest % t.shape[1]
            tok = rest // t.shape[1]
            t[tok, head, col] = 10.0 * torch.randn((n_out,), generator=g, device=device)
    if w.dtype == "fp8":
        sig = torch.randint(0, 2, (w.D,), generator=g, device=device, dtype=torch.int32) * 2 - 1
        out["sigma"] = sig.to(torch.int8)
    out["q"], out["k"], out["v"] = q.to(dt), k.to(dt), v.to(dt)
    if w.backward:
        out["do"] = torch.randn((Tq, w.H, w.D), generator=g, device=device, dtype=torch.float32).to(dt)
    if w.page_size:
        out.update(paged_cache(out["k"], out["v"], [w.Sk] * w.B, w.page_size, seed))
    return out


def paged_cache(k, v, lengths, page_size, seed, spare_pages=0):
    """The keys and values of packed sequences (``[tokens, H, D]``, lengths
    ``lengths``) laid out in a cache of ``page_size``-key pages in a seeded
    random order: returns k_cache, v_cache ``[num_pages, page_size, H, D]``,
    block_table int32 ``[B, max_pages]`` and seqlens_k int32 ``[B]``. A last
    page's rows past its sequence are zero. Pure data movement."""
    B = len(lengths)
    pages_per = [(L + page_size - 1) // page_size for L in lengths]
    num_pages = sum(pages_per) + spare_pages
    max_pages = max(max(pages_per), 1)
    perm = torch.randperm(num_pages, generator=_gen(seed, "cpu"))
    H, D = k.shape[1], k.shape[2]
    kc = torch.zeros((num_pages, page_size, H, D), dtype=k.dtype, device=k.device)
    vc = torch.zeros_like(kc)
    table = torch.zeros((B, max_pages), dtype=torch.int32)
    nxt, start = 0, 0
    for b, L in enumerate(lengths):
        n = pages_per[b]
        pages = perm[nxt:nxt + n]
        nxt += n
        table[b, :n] = pages.to(torch.int32)
        full = L // page_size
        dev_pages = pages.to(k.device)
        if full:
            kc[dev_pages[:full]] = k[start:start + full * page_size].reshape(full, page_size, H, D)
            vc[dev_pages[:full]] = v[start:start + full * page_size].reshape(full, page_size, H, D)
        rest = L - full * page_size
        if rest:
            kc[dev_pages[full], :rest] = k[start + full * page_size:start + L]
            vc[dev_pages[full], :rest] = v[start + full * page_size:start + L]
        start += L
    return {"k_cache": kc, "v_cache": vc, "block_table": table.to(k.device),
            "seqlens_k": torch.tensor(lengths, dtype=torch.int32, device=k.device)}


def sample_rows(w: Workload, inputs, n_target=2048, seed=12345):
    """Deterministic sample of (seq, head, i) query rows for large problems.

    Always includes rows 0, 127, 128, 255, 256 and the last row of every
    (seq, head) (where they exist) plus, for varlen, the first and last row of
    every sequence; the rest are uniform draws to reach ~n_target rows.
    """
    g = torch.Generator().manual_seed(seed)
    if w.varlen:
        lens = [int(x) for x in inputs["lengths"]]
    else:
        lens = [w.Sq] * w.B
    rows = set()
    for b, L in enumerate(lens):
        for h in range(w.H):
            for i in (0, 127, 128, 255, 256, L - 1):
                if 0 <= i < L:
                    rows.add((b, h, i))
    pairs = [(b, h) for b in range(len(lens)) for h in range(w.H) if lens[b] > 0]
    need = max(0, n_target - len(rows))
    if need:
        pi = torch.randint(0, len(pairs), (need,), generator=g).tolist()
        u = torch.rand((need,), generator=g).tolist()
        for p, x in zip(pi, u):
            b, h = pairs[p]
            rows.add((b, h, min(lens[b] - 1, int(x * lens[b]))))
    return sorted(rows)
