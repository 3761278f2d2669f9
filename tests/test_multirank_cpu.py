"""The N > 1 path of bench.py on the CPU, world size 2 over gloo: ranks are
independent replicas (no collective on the data path); the process group only
carries the barrier and the max-over-ranks reduction of the timing, and rank 0
alone prints the JSON line."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _cpu_env():
    env = dict(os.environ)
    env["CUDA_VISIBLE_DEVICES"] = ""
    env["OMP_NUM_THREADS"] = "2"
    return env


def test_reference_arm_two_ranks():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, env=_cpu_env(), capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout                      # rank 0 only
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


_WORKER = r"""
import os, sys, json
sys.path.insert(0, sys.argv[1])
import torch
import bench
world, rank, _ = bench.dist_setup()
dist = bench.dist_init(world, "gloo")
dist.barrier()
got = bench.max_over_ranks(1.5 + rank, world, torch.device("cpu"))
print(json.dumps({"rank": rank, "max": got}))
dist.destroy_process_group()
"""


def test_max_over_ranks_gloo(tmp_path):
    script = tmp_path / "worker.py"
    script.write_text(_WORKER)
    port = str(_free_port())
    procs = []
    for rank in range(2):
        env = _cpu_env()
        env.update({"WORLD_SIZE": "2", "RANK": str(rank), "LOCAL_RANK": str(rank),
                    "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": port})
        procs.append(subprocess.Popen([sys.executable, str(script), ROOT], cwd=ROOT, env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    assert all(o["max"] == pytest.approx(2.5) for o in outs)
