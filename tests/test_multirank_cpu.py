"""The benchmark's multi-rank path on CPU: two ranks over gloo.

bench.py runs one independent replica per GPU under torchrun (the path has no
cross-GPU exchange): every rank times its own steps, the job time is the max
over ranks, the job throughput counts every rank's units, and rank 0 alone
prints. These tests run that logic with world_size 2 on the gloo backend,
without a GPU."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


RANK_SCRIPT = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import bench
r = bench.Ranks()
local_s = 1.0 + r.rank          # rank 1 is the slow one
s = r.max(local_s)
r.barrier()
print(json.dumps({"rank": r.rank, "world": r.world, "pg": r.pg, "max_s": s,
                  "rate": bench.job_rate(r.world, 100.0, s)}), flush=True)
r.close()
"""


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_rate():
    port = free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                   WORLD_SIZE="2", LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_SCRIPT, ROOT], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["world"] == 2 and o["pg"]
        assert o["max_s"] == 2.0                 # the max over ranks, seen by both
        assert o["rate"] == pytest.approx(100.0)  # 2 ranks x 100 units / 2 s
    assert sorted(o["rank"] for o in outs) == [0, 1]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, False, "cpu") == 3.5
    assert bench.job_rate(1, 10.0, 4.0) == 2.5


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    """--impl reference under torchrun with two gloo ranks: rank 0 times the
    oracle and prints one JSON line; rank 1 exits 0 without work."""
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-3000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
