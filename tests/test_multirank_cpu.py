"""The N > 1 path of bench.py on CPU: two ranks over gloo.

The (b,h) problems are independent, so N GPUs run N replicas of the
per-GPU workload; the only collective is the barrier and the maximum of the
timed region over ranks.  These tests run that host-side logic with two
CPU processes (gloo), and the reference arm under torchrun, where rank 0
alone prints its JSON line.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # each rank reports its own "elapsed time"; every rank gets the maximum
    got = bench.max_over_ranks(10.0 + rank, w)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": got}, f)
    bench.barrier(w)
    dist.destroy_process_group()


def test_barrier_and_max_over_ranks_two_ranks(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        with open(tmp_path / f"rank{r}.json") as f:
            assert json.load(f)["max"] == 10.0 + world - 1


def test_reference_arm_under_torchrun_prints_once():
    """torchrun with two ranks: rank 0 prints one JSON line, rank 1 exits 0
    without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny_f32_fwd",
           "--gpus", "2", "--steps", "1", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="1", PYTHONPATH=ROOT)
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
