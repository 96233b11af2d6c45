"""CPU tests of bench.py's host-side pieces that the GPU runs depend on: the
oracle samples behind cpu_baseline and the reference arm, the exact FLOP
count of visible pairs, and the traffic file's digest check."""
import os
import sys
from dataclasses import replace

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from exact_attention_forward_tiled_gb300 import accounting as A  # noqa: E402
from exact_attention_forward_tiled_gb300 import workloads  # noqa: E402


def test_oracle_sample_counts_visible_pairs_with_unequal_lengths():
    # a paged-shaped workload: 16 queries at the end of 48 keys (bottom-right causal)
    w = replace(workloads.WORKLOADS["p1"], B=1, H=1, Sq=16, Sk=48, page_size=0)
    inp = workloads.make_inputs(w)
    r = bench.oracle_sample(w, {"q": inp["q"], "k": inp["k"], "v": inp["v"], "cu_seqlens_q": None}, seconds=0.0)
    assert r["rows"] == 16 and r["value"] > 0
    # the same count the GPU metric uses
    assert A.visible_pair_flops(1, w.D, [16], [48], True) == 4.0 * w.D * sum(i + 48 - 16 + 1 for i in range(16))


def test_oracle_bwd_sample_runs_on_a_small_square():
    w = replace(workloads.WORKLOADS["b1"], B=1, H=2, Sq=64, Sk=64)
    inp = workloads.make_inputs(w)
    r = bench.oracle_bwd_sample(w, inp, seconds=0.0, rows=32)
    assert r["rows"] == 32 and r["value"] > 0 and r["kind"] == "oracle"


def test_traffic_is_reported_only_for_the_current_sources(tmp_path, monkeypatch):
    digest = bench.csrc_digest()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "ncu_traffic.txt").write_text(
        f"kernel=k workload=w csrc={digest} dram_bytes_per_launch=123\n"
        f"kernel=k workload=old csrc=0000000000000000 dram_bytes_per_launch=456\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.committed_traffic("k", "w") == 123.0
    assert bench.committed_traffic("k", "old") is None
    assert bench.committed_traffic("other", "w") is None
