"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

Each rank of a replicated run times its own batch; the job's time is the slowest
rank's and its throughput counts every rank's FLOPs (weak scaling).  The
reference arm runs on rank 0 only.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, os, sys
sys.path.insert(0, os.environ["FGF8_ROOT"])
import torch.distributed as dist
dist.init_process_group("gloo")
import bench
world, rank, local = bench._dist()
t = bench._max_over_ranks(10.0 + 5.0 * rank, world, "cpu")
print(json.dumps({"rank": rank, "world": world, "local": local, "t": t,
                  "value": bench._job_tflops(4, world, t)}))
dist.destroy_process_group()
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_ranks_report_the_slowest_time():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                   WORLD_SIZE="2", LOCAL_RANK=str(rank), FGF8_ROOT=ROOT)
        procs.append(subprocess.Popen([sys.executable, "-c", CHILD], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    import bench
    expect_t = 15.0                                   # rank 1's 15 ms, not rank 0's 10 ms
    expect_v = bench.FLOPS_PER_STEP * 4 * 2 / (expect_t * 1e-3) / 1e12
    for o in outs:
        assert o["world"] == 2 and o["local"] == o["rank"]
        assert o["t"] == expect_t
        assert o["value"] == pytest.approx(expect_v, rel=1e-12)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench._max_over_ranks(7.5, 1, "cpu") == 7.5
    assert bench._job_tflops(2, 1, 1.0) == pytest.approx(bench.FLOPS_PER_STEP * 2 / 1e-3 / 1e12)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import argparse
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(steps=1, warmup=3, cpu_rows=8, ref_seconds=1.0)
    bench.run_reference(args)                          # returns at once: no oracle work, no output
    assert capsys.readouterr().out == ""
