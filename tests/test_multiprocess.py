"""The bench's multi-process path (one process per GPU under torchrun) on CPU:
gloo process groups of two ranks, no GPU.  The data path has no collective
(replicas only); what is shared is the barrier and the max over ranks of the
timed region, and rank 0 alone prints."""
import json
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


def _env():
    env = dict(os.environ)
    env["CUDA_VISIBLE_DEVICES"] = ""  # force the gloo branch of the bench's setup
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    return env


def test_reduce_max_and_barrier_over_two_gloo_ranks(tmp_path):
    out = tmp_path / "out"
    out.mkdir()
    script = (
        "import os, sys, bench\n"
        "world, rank, local = bench.dist_setup()\n"
        "assert world == 2\n"
        "bench.barrier(world)\n"
        "m = bench.reduce_max(float(rank) + 0.5, world)\n"
        f"open(os.path.join({str(out)!r}, 'rank%d' % rank), 'w').write('RANK %d MAX %s' % (rank, m))\n"
        "import torch.distributed as dist\n"
        "dist.destroy_process_group()\n"
    )
    path = tmp_path / "ranks.py"
    path.write_text(script)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), str(path)]
    r = subprocess.run(cmd, cwd=ROOT, env=_env(), capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = sorted((out / f).read_text() for f in ("rank0", "rank1"))
    assert lines == ["RANK 0 MAX 1.5", "RANK 1 MAX 1.5"]


def test_reference_arm_prints_once_under_torchrun():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--workload", "tiny", "--steps", "1", "--warmup", "3", "--gpus", "2"]
    r = subprocess.run(cmd, cwd=ROOT, env=_env(), capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
