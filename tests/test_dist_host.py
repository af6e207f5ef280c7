"""The multi-process host logic of bench.py on CPU: two gloo ranks (replicas,
no data-path collective) agree on the slowest rank's time, the whole-job
value counts every replica, and under the reference arm only rank 0 works."""
from __future__ import annotations

import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


_WORKER = r"""
import os, sys, json
sys.path.insert(0, os.environ["ROOT"])
import torch.distributed as dist
import bench
world, rank, local = bench.dist_info()
dist.init_process_group("gloo", init_method="env://", world_size=world, rank=rank)
t = bench.max_over_ranks(dist, 1.0 + 0.5 * rank)           # rank 1 is the slow one
v = bench.whole_job_gbs(world, 10**9, 4, t)
dist.barrier()
print(json.dumps({"rank": rank, "t": t, "v": v}), flush=True)
dist.destroy_process_group()
"""


def _launch(code, world, port, extra_env=None):
    procs = []
    for rank in range(world):
        env = dict(os.environ, ROOT=ROOT, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                   WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank))
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=120)
        except subprocess.TimeoutExpired:
            p.kill()
            raise
        assert p.returncode == 0, err
        outs.append(out)
    return outs


def test_two_gloo_ranks_take_the_slowest_time():
    import json
    outs = _launch(_WORKER, 2, _free_port())
    got = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert {g["rank"] for g in got} == {0, 1}
    for g in got:
        assert g["t"] == 1.5                                   # max over ranks, on every rank
        assert abs(g["v"] - 2 * 1e9 * 4 / 1.5 / 1e9) < 1e-9     # both replicas' bytes


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 0.25) == 0.25
    assert bench.whole_job_gbs(1, 2 * 10**9, 3, 2.0) == 3.0


def test_reference_arm_only_rank_zero_works():
    code = ("import sys, os; sys.path.insert(0, os.environ['ROOT']); import bench; "
            "sys.exit(bench.main(['--impl', 'reference', '--steps', '1', '--warmup', '0']))")
    env = dict(os.environ, ROOT=ROOT, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
