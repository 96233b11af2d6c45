"""Host check of the scheduler-slot table (fa::SlotTable in
csrc/sched_slots.h) that keeps two launches in flight from sharing a pair of
tile-scheduler counters. Compiled with the host compiler; no GPU."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "exact_attention_forward_tiled_gb300", "csrc")


def test_slot_table(tmp_path):
    if shutil.which("g++") is None:
        pytest.skip("needs g++")
    exe = str(tmp_path / "slot_table_check")
    subprocess.run(["g++", "-std=c++17", "-O1", "-Wall", "-I", CSRC,
                    os.path.join(HERE, "host_helpers", "slot_table_check.cpp"), "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout
