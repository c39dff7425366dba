"""The multi-rank host logic of bench.py on CPU: two gloo ranks run the replica set-up, the
barrier, the max and the sum over ranks, and the reference arm's rank gating (rank 0 alone
works)."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r"""
import json, os, sys, types
sys.path.insert(0, ROOT)
import bench
args = types.SimpleNamespace(gpus=2, steps=1, warmup=0, layers=1)
world, rank, local = bench.dist_setup(args)
bench.barrier(world)
mx = bench.max_over_ranks(1.5 + rank, world)
sm = bench.sum_over_ranks(1.0 + rank, world)
bench.barrier(world)
import torch.distributed as dist
dist.destroy_process_group()
print(json.dumps({"rank": rank, "world": world, "local": local, "max": mx, "sum": sm}), flush=True)
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_reduce_like_the_bench():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), OSCAR_DIST_BACKEND="gloo")
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_SCRIPT.replace("ROOT", repr(ROOT))], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["world"] == 2 and o["max"] == 2.5 and o["sum"] == 3.0
    assert sorted(o["rank"] for o in outs) == [0, 1]


def test_reference_arm_runs_on_rank_zero_only():
    import types
    sys.path.insert(0, ROOT)
    import bench
    args = types.SimpleNamespace(gpus=2, steps=1, warmup=0, layers=1)
    assert bench.run_reference(args, 2, 1) == 0   # returns at once: no oracle work, no output
