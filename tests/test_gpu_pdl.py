"""Launch-mode independence: a forward+backward step gives byte-identical outputs whether the
library's kernels are launched one after the other (LIGER_MOE_PDL=0), with programmatic dependent
launch (LIGER_MOE_PDL=1: each kernel may start while the previous one finishes, and waits on it
before touching memory), or in the default mode (programmatic launch for the calls below 4096
routed rows only), and whether the step runs call by call or as a replayed CUDA graph.

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
    "pdl_T256_H256_I128_E8_k2",            # below 4096 rows: programmatic launch by default
]


def _digests(workload: str, pdl, *extra: str) -> dict:
    """pdl: True (LIGER_MOE_PDL=1), False (=0) or None (unset: the default mode)."""
    env = dict(os.environ)
    env.pop("LIGER_MOE_PDL", None)
    if pdl is not None:
        env["LIGER_MOE_PDL"] = "1" if pdl else "0"
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "layer_digest.py"), workload, *extra], env=env,
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.mark.parametrize("workload", WORKLOADS)
def test_outputs_do_not_depend_on_launch_mode(workload):
    on, off, default = _digests(workload, True), _digests(workload, False), _digests(workload, None)
    for run in (on, off, default):
        assert run["device_error"] == 0
        assert run["graph"] == run["eager"], "graph replay differs from call-by-call launches"
    assert on["eager"] == off["eager"], "programmatic dependent launch changed an output"
    assert default["eager"] == off["eager"], "the default launch mode changed an output"


def test_first_call_inside_a_capture_matches():
    """No side stream exists yet when the first backward is captured: it runs in order, same bytes."""
    workload = WORKLOADS[0]
    first = _digests(workload, False, "capture_first")
    assert first["device_error"] == 0
    assert first["graph"] == _digests(workload, False)["eager"]
