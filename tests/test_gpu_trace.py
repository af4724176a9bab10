"""The library's kernel trace: one interval per kernel, or per GEMM that runs as two launches.

A GEMM that takes the heavy / light split (heavy experts as 2-SM pairs in one launch, the rest
one CTA per tile in a second) is one traced interval holding two kernel launches, and so is a
weight-gradient GEMM whose experts with many rows take the fp16 pass in a launch of their own, and
the dH GEMM of such a backward (its fp16 pass, then the refill or, with no such expert, the plain
dH); every other interval holds one.  A skewed batch of 8192 routed rows splits the forward GEMMs and
dX; a skewed batch of 32768 rows runs both weight-gradient GEMMs in an fp16 and a hi / lo launch;
a small batch whose weight-gradient blocks pair up splits dW_down.  The bench's launch count is
the sum.
"""
import pytest
import torch

import mixture_experts_routed_router_gb300 as moe
import synthetic
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu



def _step(wl, inp):
    ids, w = moe.route_topk(to_dev(inp["logits"]), wl.k)
    x, wgu, wd = to_dev(inp["x"]), to_dev(inp["wgu"]), to_dev(inp["wd"])
    d = moe.dispatch(ids, w, x, wl.E)
    h, gu, y_perm = moe.grouped_swiglu_fwd(d["x_perm"], d["m_indptr"], wgu, wd, d["w_perm"])
    moe.combine(y_perm, d["slot_to_row"], wl.T, wl.k)
    moe.bwd_dx_dw(to_dev(inp["dy"]), d["x_perm"], h, gu, ids, w, d["m_indptr"], d["row_to_slot"],
                  d["slot_to_row"], d["w_perm"], wgu, wd)


@pytest.mark.parametrize("wl,split", [
    (synthetic.Workload("split_zipf_T1024_H320_I192_E64_k8", 1024, 320, 192, 64, 8, zipf_s=1.2, router_std=0.05),
     {"gemm_gate_up_swiglu", "gemm_down_scale", "gemm_bwd_dx"}),
    (synthetic.Workload("f16_zipf_T4096_H320_I192_E64_k8", 4096, 320, 192, 64, 8, zipf_s=1.2, router_std=0.05),
     {"gemm_bwd_dh", "gemm_bwd_dw_gate_up", "gemm_bwd_dw_down"}),
    (synthetic.Workload("tiny_T256_H256_I128_E8_k2", 256, 256, 128, 8, 2), {"gemm_bwd_dw_down"}),
], ids=["skewed", "fp16", "small"])
def test_trace_intervals_count_their_launches(wl, split):
    inp = synthetic.make_inputs(wl)
    _step(wl, inp)  # side streams and kernel attributes are set up outside the traced step
    torch.cuda.synchronize()
    moe.trace_enable(True)
    try:
        _step(wl, inp)
        torch.cuda.synchronize()
        records = moe.trace_records()
        counts = moe.trace_launch_counts()
    finally:
        moe.trace_enable(False)
    assert moe.device_error() == 0
    assert len(records) == len(counts) > 0
    for (name, ms), n in zip(records, counts):
        assert ms > 0.0, name
        assert n == (2 if name in split else 1), (name, n)
    assert {name for name, _ in records} >= split
