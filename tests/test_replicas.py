"""The benchmark's N > 1 path on the CPU: two gloo ranks check the
max-over-ranks time and the whole-job rate, and the reference arm under two
ranks prints one line from rank 0 while rank 1 exits quietly.  (Every GPU
box here has one GPU, so the path shards as independent replicas and has no
collective in its data path; only the timing reduction crosses ranks.)"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import os, sys
sys.path.insert(0, {root!r})
import torch, torch.distributed as dist
import bench
dist.init_process_group("gloo", init_method="tcp://127.0.0.1:{port}", rank=int(sys.argv[1]), world_size=2)
r = dist.get_rank()
t = bench.max_over_ranks(10.0 + 5.0 * r, 2)       # rank 1 is the slower replica
v = bench.job_throughput(100.0, 4, 2, t)            # 100 units per rank-step
print(r, t, v, flush=True)
dist.destroy_process_group()
"""


def test_max_over_ranks_and_job_rate_gloo(tmp_path):
    pytest.importorskip("torch.distributed")
    script = tmp_path / "worker.py"
    script.write_text(WORKER.format(root=ROOT, port=free_port()))
    procs = [subprocess.Popen([sys.executable, str(script), str(r)], stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                              text=True) for r in range(2)]
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    for r, (o, _) in enumerate(outs):
        rank, t, v = o.split()
        assert int(rank) == r
        assert float(t) == 15.0                              # the max, on every rank
        assert abs(float(v) - 100.0 * 4 * 2 / 0.015) < 1e-6  # all ranks' units over the max time


def test_reference_arm_under_two_ranks():
    env = dict(os.environ, MASTER_ADDR="127.0.0.1")
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--ref-sample", "0.005"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2
    assert res["e2e"]["h2d_bytes_per_step"] == 0 and res["cpu_baseline"]["kind"] == "oracle"


def test_gpus_flag_starts_that_many_ranks():
    """`bench.py --gpus 2` started as a plain process launches its two ranks
    itself (one per GPU) and prints one line for the whole job."""
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3", "--ref-sample", "0.005"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    assert json.loads(lines[0])["n_gpus"] == 2


def test_gpus_flag_must_match_world_size():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=120, env=env, cwd=ROOT)
    assert r.returncode != 0 and "WORLD_SIZE" in r.stderr
