"""The N > 1 host path of bench.py, on CPU: two gloo ranks (127.0.0.1) run
the replicas' rank logic -- barrier, max over ranks of the step time, the
whole-job value -- and only rank 0 prints the reference line."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import bench
world = int(os.environ["WORLD_SIZE"]); rank = int(os.environ["RANK"])
bench.init_ranks(world)
bench.barrier(world)
ms = bench.max_over_ranks(2.0 + rank, world)          # rank 1 is the slow replica
value = bench.job_value(1e9, ms, world)
print(json.dumps({{"rank": rank, "ms": ms, "value": value}}), flush=True)
import torch.distributed as dist
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_ranks(code, world=2, extra_env=None):
    port = _free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                   RANK=str(rank), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(out)
    return outs


def test_two_gloo_ranks_take_the_slowest_step_time():
    outs = _run_ranks(WORKER.format(root=ROOT))
    lines = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert all(l["ms"] == 3.0 for l in lines)                     # max over ranks
    assert all(abs(l["value"] - 2 * 1e9 / 3e-3) < 1 for l in lines)  # both ranks' units / slowest time


def test_reference_arm_prints_on_rank_zero_only():
    """Under torchrun the oracle arm runs on rank 0 alone; rank 1 exits 0
    without output."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny_bf16",
           "--steps", "1", "--warmup", "1"]
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env["RANK"] = "0"
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
