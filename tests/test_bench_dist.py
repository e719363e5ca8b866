"""The multi-process path of bench.py on CPU: two gloo ranks exchange the
barrier and the max-over-ranks timing, the whole-job rate counts every rank's
units over the slowest rank's time, and the reference arm runs on rank 0 only."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r"""
import json, os, sys, time
sys.path.insert(0, sys.argv[1])
import torch
import bench
d = bench.Dist(torch, backend="gloo")
rank = d.rank
d.barrier()
elapsed = 0.5 + rank           # rank 1 is the slow one
m = d.max(elapsed)
d.barrier()
out = {"rank": rank, "world": d.world, "max": m, "rate": bench.job_rate(d.world, 10, 1_000_000_000, m)}
print(json.dumps(out), flush=True)
d.close()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_ranks(code_args, world=2, timeout=120):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(world),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, *code_args], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            o, e = p.communicate(timeout=timeout)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            raise
        assert p.returncode == 0, e[-2000:]
        outs.append(o)
    return outs


def test_two_gloo_ranks_agree_on_the_max_and_the_job_rate():
    pytest.importorskip("torch")
    outs = _run_ranks(["-c", RANK_SCRIPT, ROOT])
    res = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert sorted(r["rank"] for r in res) == [0, 1]
    for r in res:
        assert r["world"] == 2
        assert r["max"] == 1.5                      # the slowest rank decides
        assert abs(r["rate"] - 2 * 10 / 1.5) < 1e-9  # both ranks' units over that time


def test_single_process_needs_no_process_group():
    torch = pytest.importorskip("torch")
    sys.path.insert(0, ROOT)
    import bench

    d = bench.Dist(torch, backend="gloo")
    assert d.world == int(os.environ.get("WORLD_SIZE", "1")) and d.pg is None
    assert d.max(3.25) == 3.25
    assert bench.job_rate(1, 4, 2_000_000_000, 2.0) == 4.0


def test_reference_arm_runs_on_rank_zero_only():
    """Rank 1 of the reference arm exits 0 without work or output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""
