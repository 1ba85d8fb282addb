"""The multi-GPU path on CPU: two gloo ranks.

The scan shards by batch with no data-path collective (each rank scans its own
sequences); what runs across ranks is the benchmark's host logic: the rendezvous, the
barrier, the slowest-rank timing (an all-reduce of the step time with MAX) and rank 0
alone printing the line.  These tests run that logic as two real processes.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist, w, r, local = bench.dist_setup()
    assert dist.get_backend() == "gloo"
    bench.barrier(dist)
    slowest = bench.max_over_ranks(dist, 10.0 * (r + 1))
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "max": slowest}, f)
    dist.destroy_process_group()


def test_slowest_rank_time_over_gloo(tmp_path):
    port = free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert [x["rank"] for x in res] == [0, 1]
    assert all(x["world"] == 2 for x in res)
    assert all(x["max"] == 20.0 for x in res)  # every rank sees the slowest rank's time


def test_reference_arm_under_torchrun_prints_one_line():
    """Launched the way a multi-GPU bench run is (torchrun, 2 ranks, 127.0.0.1): rank 0 times
    the oracle and prints one line; rank 1 does no work and exits 0."""
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "1", "--workload", "c0"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
