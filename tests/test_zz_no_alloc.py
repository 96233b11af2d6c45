"""The allocation-free split-KV entry point, for callers that cannot allocate
device memory (no cudaMalloc where they run, or an allocator that must not
grow): it must give what the workspace-taking entry point gives.

Collected last on purpose, so a run that stops at the first failure has run
every other test first. It also passes on its own in a fresh process.
"""
import pytest
import torch

from exact_attention_forward_tiled_gb300 import api
from exact_attention_forward_tiled_gb300 import build as fa_build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    fa_build.build()
    api.lib()


def _rand(shape, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)


def test_noalloc_matches_workspace_entry_point_twice():
    """Two calls in a row (different inputs, different key ranges) through the
    C ABI match fa_fwd_splitkv with a caller workspace within the bf16 bars
    of the other tests (max |dO| <= 1e-2, |dLSE| <= 1e-3)."""
    for call, (B, H, Sq, Sk, D, causal, splits) in enumerate([(2, 4, 256, 4096, 128, False, 0),
                                                              (1, 3, 100, 2049, 64, True, 5)]):
        q = _rand((B * Sq, H, D), 10 * call + 1)
        k = _rand((B * Sk, H, D), 10 * call + 2)
        v = _rand((B * Sk, H, D), 10 * call + 3)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, Sq), device="cuda")
        api.fa_fwd_splitkv_noalloc(q, k, v, o, lse, B, H, Sq, Sk, D, D ** -0.5, causal, splits)
        api.fa_get_device_status()
        o_ref, lse_ref = api.attention_forward_splitkv(q, k, v, batch=B, causal=causal, num_splits=splits)
        api.fa_get_device_status()
        assert (o.float() - o_ref.float()).abs().max().item() <= 1e-2, call
        assert (lse - lse_ref).abs().max().item() <= 1e-3, call


def test_noalloc_rejects_problems_beyond_its_scratch():
    """A problem whose scratch would exceed the built-in array is refused up
    front with FA_ERR_SCRATCH_LIMIT; no pointer is touched."""
    B, H, Sq, Sk, D = 1, 64, 8192, 8192, 256
    need = api.fa_fwd_splitkv_workspace_size(B, H, Sq, Sk, D, 16)
    assert need > 64 << 20
    t = torch.empty((16, 1, 256), device="cuda", dtype=torch.bfloat16)
    lse = torch.empty((1,), device="cuda")
    st = api.fa_fwd_splitkv_noalloc(t, t, t, t, lse, B, H, Sq, Sk, D, 0.0625, 0, 16, check=False)
    assert st == -8
    assert "scratch" in api.strerror(st)


def test_noalloc_near_its_limit():
    """A problem whose scratch is just under the 64 MiB array (63 key ranges
    of 1 MiB of partial O each; the partial LSE then sits in the last MiB):
    the same result as fa_fwd_splitkv with a caller workspace."""
    B, H, Sq, Sk, D, splits = 1, 8, 256, 8000, 128, 63
    need = api.fa_fwd_splitkv_workspace_size(B, H, Sq, Sk, D, splits)
    assert (63 << 20) < need <= (64 << 20), need
    q = _rand((B * Sq, H, D), 31)
    k = _rand((B * Sk, H, D), 32)
    v = _rand((B * Sk, H, D), 33)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Sq), device="cuda")
    api.fa_fwd_splitkv_noalloc(q, k, v, o, lse, B, H, Sq, Sk, D, D ** -0.5, True, splits)
    api.fa_get_device_status()
    o_ref, lse_ref = api.attention_forward_splitkv(q, k, v, batch=B, causal=True, num_splits=splits)
    api.fa_get_device_status()
    assert (o.float() - o_ref.float()).abs().max().item() <= 1e-2
    assert (lse - lse_ref).abs().max().item() <= 1e-3
