"""Multi-GPU host logic on CPU: two gloo ranks run the benchmark's
replica bookkeeping (barrier, max over ranks, aggregate images/s) and the
reference arm under torchrun-style environment variables.  No GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r'''
import os, sys, json
sys.path.insert(0, sys.argv[1])
import torch, torch.distributed as dist
import bench
rank = int(os.environ["RANK"]); world = int(os.environ["WORLD_SIZE"])
dist.init_process_group("gloo")
bench.barrier(dist)
t = bench.max_over_ranks(dist, 10.0 + 5.0 * rank, "cpu")   # ranks took 10 and 15 ms
agg = bench.aggregate_images_per_s(world, 256, 100, t)
if rank == 0:
    print(json.dumps({"max_ms": t, "value": agg}))
dist.destroy_process_group()
'''


def _env(rank, world, port):
    env = dict(os.environ)
    env.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    return env


def _free_port():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_two_rank_max_and_aggregate():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", WORKER, ROOT], env=_env(r, 2, port), stdout=subprocess.PIPE,
                              stderr=subprocess.PIPE, text=True) for r in range(2)]
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    line = json.loads(outs[0][0].strip().splitlines()[-1])
    assert line["max_ms"] == 15.0
    # both ranks' images over the slowest rank's time
    assert abs(line["value"] - 2 * 256 * 100 / 0.015) < 1e-6 * line["value"]
    assert outs[1][0].strip() == ""


def test_reference_arm_prints_once_under_two_ranks():
    port = _free_port()
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "3",
           "--warmup", "1", "--cpu-seconds", "1"]
    procs = [subprocess.Popen(cmd, env=_env(r, 2, port), stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True,
                              cwd=ROOT) for r in range(2)]
    outs = [p.communicate(timeout=300) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    lines = [l for l in outs[0][0].splitlines() if l.startswith("{")]
    assert len(lines) == 1 and outs[1][0].strip() == ""
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "images/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
