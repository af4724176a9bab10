"""bench.py with N > 1 ranks, on CPU: two processes launched by torch.distributed.run.

N GPUs run N independent replicas of the layer step: the path has no exchange step on one
GPU's data.  So the ranks meet only around the timed region: a barrier on both sides, the
slowest rank's time, and the whole-job rate computed from it.  Here that host logic runs over
gloo with world size 2.  The reference arm is launched the same way; rank 0 alone runs the
oracle and prints one line, and the other rank exits 0 without work.
"""
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


def _torchrun(*args: str, timeout: int = 300) -> subprocess.CompletedProcess:
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), *args]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    return subprocess.run(cmd, capture_output=True, text=True, timeout=timeout, cwd=ROOT, env=env)


def _json_lines(text: str) -> list[dict]:
    return [json.loads(line) for line in text.splitlines() if line.startswith("{")]


def test_ranks_agree_on_the_slowest_time_and_the_whole_job_rate():
    r = _torchrun(os.path.join("tests", "ranks_probe.py"))
    assert r.returncode == 0, r.stderr[-3000:]
    lines = sorted(_json_lines(r.stdout), key=lambda d: d["rank"])
    assert [d["rank"] for d in lines] == [0, 1]
    for d in lines:
        assert d["world"] == 2
        assert d["slowest_ms"] == 20.0                 # rank 1's time, on both ranks
        assert d["rate"] == pytest.approx(2 * 1000.0 / 0.020)  # both ranks' units over the slowest time


def test_whole_job_rate_is_units_of_all_ranks_over_the_slowest_time():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.whole_job_rate(1, 500.0, 250.0) == pytest.approx(2000.0)
    assert bench.whole_job_rate(4, 500.0, 250.0) == pytest.approx(8000.0)
    assert bench.rank_max(3.5, None, "cpu") == 3.5  # one rank: no process group, the value itself


def test_reference_arm_prints_once_from_rank_zero():
    r = _torchrun("bench.py", "--impl", "reference", "--gpus", "2", "--workload", "tiny_T256_H256_I128_E8_k2",
                  "--steps", "1", "--warmup", "0", timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1, r.stdout[-2000:]
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
