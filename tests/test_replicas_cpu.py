"""Multi-process (world size 2, gloo, CPU) checks of the replicas path of bench.py.

The MoE layer does not shard across GPUs here: each rank runs its own batch
and nothing crosses ranks on the data path.  What does cross ranks is the
timing protocol (a barrier on both sides of the timed region, the maximum of
the per-rank times) and the rule that only rank 0 runs the host reference arm
and prints.  These tests run that protocol as two gloo processes.
"""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


_RANK_SCRIPT = r"""
import argparse, json, sys
sys.path.insert(0, {root!r})
import bench
import torch.distributed as dist
rank, world, local = bench.dist_init()
bench.barrier(world)
# each rank reports a different time; all must agree on the slowest
t = bench.max_over_ranks(0.25 + rank, world)
ref = bench.run_reference(argparse.Namespace(tokens=64, ref_tokens=4, warmup=0, steps=1), rank, world) \
    if rank != 0 else "not run"
print(json.dumps({{"rank": rank, "world": world, "max": t, "backend": dist.get_backend(),
                  "ref_is_none": ref is None}}), flush=True)
dist.destroy_process_group()
"""


def test_dist_helpers_world2_gloo():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, WORLD_SIZE="2", RANK=str(r), LOCAL_RANK=str(r),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", _RANK_SCRIPT.format(root=ROOT)],
                                      env=env, cwd=ROOT, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=240)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    outs.sort(key=lambda d: d["rank"])
    assert [d["rank"] for d in outs] == [0, 1]
    for d in outs:
        assert d["world"] == 2
        assert d["backend"] == "gloo"
        assert d["max"] == pytest.approx(1.25)   # the slower rank's time, on every rank
    # the reference arm does no work on a rank other than 0
    assert outs[1]["ref_is_none"] is True


def test_reference_arm_torchrun_world2(oracle_lib):
    """bench.py --impl reference under torchrun: rank 0 alone prints one line; all exit 0."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--ref-tokens", "4"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 2
    assert d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle"
