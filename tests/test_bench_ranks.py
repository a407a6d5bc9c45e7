"""The bench's multi-rank path on CPU: two gloo ranks (127.0.0.1) run independent
replicas; every rank must get the slowest rank's time, and the job's rate must count the
units of all ranks over that time.  (The path does not shard: no collective but this
timing reduction.)"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, os, sys
import torch
import torch.distributed as dist
sys.path.insert(0, os.environ["K3_ROOT"])
import bench
rank = int(os.environ["RANK"])
dist.init_process_group("gloo", rank=rank, world_size=int(os.environ["WORLD_SIZE"]))
t = bench.reduce_max(dist, 1.5 + rank, torch.device("cpu"))   # rank 1 is the slow one
rate = bench.job_rate(10, dist.get_world_size(), t)
dist.barrier()
print(json.dumps({"rank": rank, "t": t, "rate": rate}), flush=True)
dist.destroy_process_group()
"""


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_take_the_slowest_time():
    port = free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), K3_ROOT=ROOT)
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    out = []
    for p in procs:
        so, se = p.communicate(timeout=120)
        assert p.returncode == 0, se[-2000:]
        out.append(json.loads(so.strip().splitlines()[-1]))
    for r in out:
        assert r["t"] == 2.5              # the slowest rank's time, on both ranks
        assert r["rate"] == 10 * 2 / 2.5  # all ranks' units over that time


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(None, 3.25, None) == 3.25
    assert bench.job_rate(7, 1, 2.0) == 3.5


def test_timed_blocks_cover_a_second_of_load():
    # the clock sampler reads every 200 ms: short timed regions are repeated (blocks of
    # exactly K steps each) until the timed work lasts at least a second
    sys.path.insert(0, ROOT)
    import bench
    assert bench.blocks_needed(0.3) == 4
    assert bench.blocks_needed(0.25) == 4
    assert bench.blocks_needed(2.0) == 1
    assert bench.blocks_needed(0.0) == 1
