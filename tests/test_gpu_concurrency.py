"""The scheduler-slot limit through the C ABI: at most 64 launches of the
library may be in flight on a device; one more is refused with FA_ERR_BUSY
(nothing is launched), and once the queue drains every slot is usable again
and the results are right."""
import numpy as np
import pytest
import torch

from exact_attention_forward_tiled_gb300 import api
from exact_attention_forward_tiled_gb300 import build as fa_build
from oracle import oracle as orc

pytestmark = pytest.mark.gpu
FA_ERR_BUSY = -9


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    fa_build.build()
    api.lib()


def test_65th_launch_in_flight_is_refused():
    # about 6 ms per launch: 65 raw calls queue on one stream far faster than
    # the first launch runs
    B, H, S, D = 16, 16, 8192, 128
    g = torch.Generator(device="cuda").manual_seed(5)
    q, k, v = (torch.randn((B * S, H, D), generator=g, device="cuda").to(torch.bfloat16) for _ in range(3))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S), device="cuda")
    import ctypes
    L = api.lib()
    args = [ctypes.c_void_p(t.data_ptr()) for t in (q, k, v, o, lse)] + [B, H, S, S, D, ctypes.c_float(D ** -0.5),
                                                                        0, None, None, 0, 0, api.FA_BF16, None]
    torch.cuda.synchronize()
    sts = [L.fa_fwd(*args) for _ in range(65)]
    assert sts[:64] == [0] * 64, sts
    assert sts[64] == FA_ERR_BUSY, sts[64]
    assert "in flight" in api.strerror(FA_ERR_BUSY)
    torch.cuda.synchronize()
    assert api.fa_get_device_status()[0] == 0
    # the queue has drained: every slot is free again
    sts = [api.fa_fwd(q, k, v, o, lse, B, H, S, S, D, D ** -0.5, False, check=False) for _ in range(3)]
    assert sts == [0, 0, 0]
    api.fa_get_device_status()
    rows = [(0, 0, 0), (3, 7, 4095), (15, 15, 8191), (9, 2, 128)]
    ref, ref_l = orc.attention_rows(q, k, v, rows, scale=D ** -0.5, causal=False, nseq=B, Sq=S, Sk=S)
    got = np.stack([o[b * S + i, h].float().cpu().numpy() for b, h, i in rows])
    assert np.abs(got - ref).max() <= 1e-2
