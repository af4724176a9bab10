"""Launch-mode independence: a forward+backward step gives byte-identical outputs whether the
library's kernels are launched one after the other (the default) or with programmatic dependent
launch (LIGER_MOE_PDL=1: each kernel may start while the previous one finishes, and waits on it
before touching memory), and whether the step runs call by call or as a replayed CUDA graph.

A kernel that read its inputs before its predecessor had finished writing them would show up
here as a digest mismatch.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORKLOADS = [
    "pdl_T4096_H512_I256_E16_k4_zipf1.2",  # 2-SM pair tiles, skewed load, empty experts
    "pdl_T512_H256_I128_E64_k8",           # few rows per expert: one-CTA and multicast tiles
]


def _digests(workload: str, pdl: bool, *extra: str) -> dict:
    env = dict(os.environ)
    env.pop("LIGER_MOE_PDL", None)
    if pdl:
        env["LIGER_MOE_PDL"] = "1"
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "layer_digest.py"), workload, *extra], env=env,
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.mark.parametrize("workload", WORKLOADS)
def test_outputs_do_not_depend_on_launch_mode(workload):
    on, off = _digests(workload, True), _digests(workload, False)
    for run in (on, off):
        assert run["device_error"] == 0
        assert run["graph"] == run["eager"], "graph replay differs from call-by-call launches"
    assert on["eager"] == off["eager"], "programmatic dependent launch changed an output"


def test_first_call_inside_a_capture_matches():
    """No side stream exists yet when the first backward is captured: it runs in order, same bytes."""
    workload = WORKLOADS[0]
    first = _digests(workload, False, "capture_first")
    assert first["device_error"] == 0
    assert first["graph"] == _digests(workload, False)["eager"]
