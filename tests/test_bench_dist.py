"""bench.py's multi-rank path on CPU: two gloo ranks on 127.0.0.1.

The timed region's length is the maximum over ranks (so `value` divides the
work of every rank by the slowest one), and under torchrun only rank 0 runs
and prints the reference arm while the other ranks exit 0 without work.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2",
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import bench
    import torch.distributed as dist
    world, r, _ = bench.dist_setup(2)
    assert (world, r) == (2, rank)
    # each rank times a different duration; every rank must see the slowest
    got = bench.max_over_ranks(1.5 * (rank + 1), world, torch.device("cpu"))
    bench.barrier(world)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": got}, f)
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    mp.start_processes(_rank_main, args=(_free_port(), str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for rank in range(2):
        with open(tmp_path / f"rank{rank}.json") as f:
            assert json.load(f)["max"] == 3.0


@pytest.mark.timeout(300)
def test_reference_arm_prints_once_under_torchrun():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "2",
           "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=280)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 2
    assert line["value"] > 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle"
