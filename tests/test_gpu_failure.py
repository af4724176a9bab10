"""Failure detection on the GPU without a fault: the bounded pipeline wait.

Every wait of the grouped-GEMM pipeline is bounded; when one runs out the kernel sets the
WAIT_TIMEOUT bit of the device error flag and returns.  liger_moe_selftest_wait_timeout makes a
wait run out on purpose (an mbarrier phase that nothing completes) with a short limit.  The test
checks that the status reaches the host and that the context keeps working afterwards.
"""
import time

import numpy as np
import pytest

import mixture_experts_routed_router_gb300 as moe
import oracle
import synthetic
from tests.gpu_util import to_dev, to_host

pytestmark = pytest.mark.gpu

WAIT_TIMEOUT = {v: k for k, v in moe.DEVERR.items()}["WAIT_TIMEOUT"]


def test_a_wait_that_runs_out_is_reported_and_the_context_survives():
    assert moe.device_error() == 0
    t0 = time.perf_counter()
    moe.selftest_wait_timeout(50_000)  # 50 ms
    flags = moe.device_error()  # synchronises the stream, reads and clears the flag
    dt = time.perf_counter() - t0
    assert flags == WAIT_TIMEOUT
    assert 0.05 <= dt < 5.0
    assert moe.device_error() == 0  # cleared
    # the next calls run normally
    wl = synthetic.WORKLOADS["tiny_T256_H256_I128_E8_k2"]
    inp = synthetic.make_inputs(wl)
    ids, w = moe.route_topk(to_dev(inp["logits"]), wl.k)
    d = moe.dispatch(ids, w, to_dev(inp["x"]), wl.E)
    h, gu, y = moe.grouped_swiglu_fwd(d["x_perm"], d["m_indptr"], to_dev(inp["wgu"]), to_dev(inp["wd"]), d["w_perm"])
    assert moe.device_error() == 0
    rids, _ = oracle.route_topk(inp["logits"], wl.k)
    np.testing.assert_array_equal(to_host(ids), rids)
    assert np.isfinite(to_host(y.float())).all()


def test_the_gemm_wait_limit_is_far_above_a_real_wait():
    """The same GEMMs complete well inside their 2 s per-wait limit (no spurious timeouts): a full
    fwd+bwd at the bench workload's per-expert load leaves the flag clear."""
    wl = synthetic.Workload("ncu_T2048_H2048_I512_E64_k8", 2048, 2048, 512, 64, 8)
    inp = synthetic.make_inputs(wl)
    ids, w = moe.route_topk(to_dev(inp["logits"]), wl.k)
    d = moe.dispatch(ids, w, to_dev(inp["x"]), wl.E)
    wgu, wd = to_dev(inp["wgu"]), to_dev(inp["wd"])
    h, gu, y = moe.grouped_swiglu_fwd(d["x_perm"], d["m_indptr"], wgu, wd, d["w_perm"])
    moe.bwd_dx_dw(to_dev(inp["dy"]), d["x_perm"], h, gu, ids, w, d["m_indptr"], d["row_to_slot"], d["slot_to_row"],
                  d["w_perm"], wgu, wd)
    assert moe.device_error() == 0
