"""The scheduler slots through the C ABI. A device has 64 pairs of
tile-scheduler counters; with 64 launches of the library in flight, the next
launch reuses the slot handed out longest ago and its stream first waits, on
the GPU, for that slot's previous launch. Deep queues on one stream and over
several streams give the right results, and a launch captured into a CUDA
graph replays correctly."""
import ctypes

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


def _inputs(B, H, S, D, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    q, k, v = (torch.randn((B * S, H, D), generator=g, device="cuda").to(torch.bfloat16) for _ in range(3))
    return q, k, v, torch.empty_like(q), torch.empty((B, H, S), device="cuda")


def _raw_args(q, k, v, o, lse, B, H, S, D, stream=None):
    return [ctypes.c_void_p(t.data_ptr()) for t in (q, k, v, o, lse)] + [
        B, H, S, S, D, ctypes.c_float(D ** -0.5), 0, None, None, 0, 0, api.FA_BF16,
        ctypes.c_void_p(stream.cuda_stream) if stream is not None else None]


def _check_rows(q, k, v, o, lse, B, S, D, rows):
    ref, ref_l = orc.attention_rows(q, k, v, rows, scale=D ** -0.5, causal=False, nseq=B, Sq=S, Sk=S)
    got = np.stack([o[b * S + i, h].float().cpu().numpy() for b, h, i in rows])
    got_l = np.array([lse[b, h, i].item() for b, h, i in rows])
    assert np.abs(got - ref).max() <= 1e-2
    assert np.abs(got_l - ref_l).max() <= 1e-3


def test_deep_queue_on_one_stream():
    # about 6 ms per launch: 200 raw calls queue on one stream far faster than
    # the launches run, so every call after the 64th reuses a held slot
    B, H, S, D = 16, 16, 8192, 128
    q, k, v, o, lse = _inputs(B, H, S, D, 5)
    L = api.lib()
    args = _raw_args(q, k, v, o, lse, B, H, S, D)
    torch.cuda.synchronize()
    sts = [L.fa_fwd(*args) for _ in range(200)]
    assert sts == [0] * 200, sts
    torch.cuda.synchronize()
    assert api.fa_get_device_status()[0] == 0
    _check_rows(q, k, v, o, lse, B, S, D, [(0, 0, 0), (3, 7, 4095), (15, 15, 8191), (9, 2, 128)])


def test_deep_queues_on_several_streams():
    # four streams, each with its own problem, 40 launches each, interleaved:
    # 160 launches in flight share the 64 slots across streams
    B, H, S, D = 4, 16, 8192, 128
    streams = [torch.cuda.Stream() for _ in range(4)]
    probs = [_inputs(B, H, S, D, 20 + i) for i in range(4)]
    L = api.lib()
    args = [_raw_args(*p, B, H, S, D, stream=s) for p, s in zip(probs, streams)]
    torch.cuda.synchronize()
    sts = []
    for _ in range(40):
        for a in args:
            sts.append(L.fa_fwd(*a))
    assert sts == [0] * 160, sts
    torch.cuda.synchronize()
    assert api.fa_get_device_status()[0] == 0
    for p in probs:
        _check_rows(*p, B, S, D, [(0, 0, 0), (1, 9, 4097), (3, 15, 8191)])


def test_launch_captured_into_a_graph():
    B, H, S, D = 2, 8, 2048, 128
    q, k, v, o, lse = _inputs(B, H, S, D, 31)
    api.fa_fwd(q, k, v, o, lse, B, H, S, S, D, D ** -0.5, False)
    torch.cuda.synchronize()
    o_eager, lse_eager = o.clone(), lse.clone()
    o.zero_()
    lse.zero_()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            st = api.fa_fwd(q, k, v, o, lse, B, H, S, S, D, D ** -0.5, False, stream=side, check=False)
    assert st == 0
    torch.cuda.synchronize()
    for _ in range(3):
        o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, o_eager) and torch.equal(lse, lse_eager)
    assert api.fa_get_device_status()[0] == 0
