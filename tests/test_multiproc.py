"""bench.py's multi-process host logic on the CPU: two gloo ranks on 127.0.0.1 through
torch.distributed.run, as the driver launches bench.py for N > 1."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _torchrun(args, timeout=240):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port())] + args
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def test_barrier_and_max_over_ranks_gloo(tmp_path):
    r = _torchrun([os.path.join("tests", "dist_bench_worker.py"), str(tmp_path)])
    assert r.returncode == 0, r.stderr[-2000:]
    res = [json.loads((tmp_path / f"rank{i}.json").read_text()) for i in range(2)]
    assert sorted(x["rank"] for x in res) == [0, 1]
    for x in res:
        assert x["world"] == 2
        assert x["max"] == 20.0      # the slowest rank's time is what the bench reports
        assert x["sum"] == 3.0


@pytest.mark.timeout(600)
def test_reference_arm_prints_once_under_torchrun():
    r = _torchrun(["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"], timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
