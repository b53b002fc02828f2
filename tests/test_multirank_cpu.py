"""The N > 1 path of bench.py on CPU: independent replicas joined only for
timing (a barrier and max/sum reductions), over gloo with world size 2."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    bench.dist_init(world, "gloo")
    # rank r processed (r+1) GB in (r+2) seconds
    total, slowest = bench.aggregate((rank + 1) * 1e9, rank + 2.0, torch.device("cpu"))
    bench.barrier()
    out[rank] = (total, slowest, bench.dist_env())
    dist.destroy_process_group()


def test_replica_aggregation_two_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for r in range(2):
        total, slowest, env = res[r]
        assert total == 3e9            # all ranks' bytes
        assert slowest == 3.0          # the slowest rank's time
        assert env[0] == r and env[1] == 2


def test_reference_arm_non_zero_rank_prints_nothing():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                        "--warmup", "0", "--workload", "single_head_l256"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_gpus_flag_must_match_the_launcher():
    env = dict(os.environ, RANK="0", WORLD_SIZE="2", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "4", "--steps", "1",
                        "--warmup", "0", "--workload", "single_head_l256"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode != 0 and "--gpus 4" in r.stderr


def test_gpus_flag_without_launcher_starts_the_ranks_itself():
    """`bench.py --gpus 2` with no launcher around it starts two ranks itself
    (torch.distributed.run on 127.0.0.1); rank 0 prints one line for both."""
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                        "--warmup", "0", "--workload", "single_head_l256"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["config"]["parallelism"] == "replicas2"


def test_single_process_aggregate_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(5.0, 2.0, torch.device("cpu")) == (5.0, 2.0)
