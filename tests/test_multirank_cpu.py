"""The N > 1 launch path of bench.py on CPU: two gloo ranks (world_size 2,
127.0.0.1 rendezvous), as torchrun would start them. The forward shards over
(batch x heads) with no data exchange, so the only cross-rank steps are the
barrier and the max-over-ranks time; the reference arm runs on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    my_ms = [1.5, 2.25][rank]
    slow = bench.max_over_ranks(my_ms)
    value = bench.job_value(2.2e12, world, slow)
    dist.barrier()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"slow": slow, "value": value}, f)
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn", join=True)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    assert res[0]["slow"] == res[1]["slow"] == 2.25        # every rank sees the slowest rank's time
    assert abs(res[0]["value"] - 2 * 2.2e12 / 2.25e-3 / 1e12) < 1e-9


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_value(1e12, 1, 1.0) == 1000.0     # 1e12 FLOP in 1 ms = 1000 TFLOP/s


def test_reference_arm_runs_on_rank0_only(tmp_path):
    """Under torchrun the reference arm's non-zero ranks exit 0 without work."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
