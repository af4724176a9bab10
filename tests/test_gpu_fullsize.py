"""Full-size parity on every workload shape, in the launch configuration the benchmark uses.

Routing ids, counts, m_indptr and both permutations are compared whole and must
be bit-exact.  Float outputs are compared on samples the oracle computes one by
one: the layer output Y, dX and d_logits of sampled tokens, h / y of sampled
rows, and the weight gradients of sampled experts (the lightest non-empty one,
a median one and the heaviest one up to a row budget).
"""
import numpy as np
import pytest
import torch

import mixture_experts_routed_router_gb300 as moe
import oracle
import synthetic
from tests.gpu_util import to_dev, to_host
from tests.helpers import assert_close, bf16_to_f64

pytestmark = pytest.mark.gpu

N_TOKENS = 24
ROW_BUDGET = 1200  # rows of the sampled experts whose dW the oracle recomputes


def _sample_experts(counts):
    nz = np.nonzero(counts)[0]
    order = nz[np.argsort(counts[nz], kind="stable")]
    picks = [order[0], order[len(order) // 2]]
    for e in order[::-1]:
        if counts[e] <= ROW_BUDGET:
            picks.append(e)
            break
    return np.unique(np.array(picks, dtype=np.int32))


@pytest.mark.parametrize("name", list(synthetic.WORKLOADS))
def test_full_size_sampled_parity(name):
    wl = synthetic.WORKLOADS[name]
    inp = synthetic.make_inputs(wl, seed=0)
    T, H, I, E, k, R = wl.T, wl.H, wl.I, wl.E, wl.k, wl.R
    logits, x, dy = to_dev(inp["logits"]), to_dev(inp["x"]), to_dev(inp["dy"])
    wgu, wd = to_dev(inp["wgu"]), to_dev(inp["wd"])

    ids, w = moe.route_topk(logits, k)
    d = moe.dispatch(ids, w, x, E)
    h, gu, y_perm = moe.grouped_swiglu_fwd(d["x_perm"], d["m_indptr"], wgu, wd, d["w_perm"])
    Y = moe.combine(y_perm, d["slot_to_row"], T, k)
    dx, dwgu, dwd, dl = moe.bwd_dx_dw(dy, d["x_perm"], h, gu, ids, w, d["m_indptr"], d["row_to_slot"],
                                      d["slot_to_row"], d["w_perm"], wgu, wd)
    assert moe.device_error() == 0

    # integer work: whole tensors, bit-exact
    rids, rw = oracle.route_topk(inp["logits"], k)
    np.testing.assert_array_equal(to_host(ids), rids)
    np.testing.assert_allclose(to_host(w), rw, rtol=2e-6, atol=1e-8)
    ref = oracle.dispatch(rids, rw, None, E)
    for key in ("counts", "m_indptr", "row_to_slot", "slot_to_row"):
        np.testing.assert_array_equal(to_host(d[key]), ref[key], err_msg=key)

    rng = np.random.default_rng(1234)
    toks = np.sort(rng.choice(T, size=min(N_TOKENS, T), replace=False)).astype(np.int32)
    rows = np.sort(rng.choice(R, size=min(64, R), replace=False)).astype(np.int32)

    # expert MLP rows (h, y) on the GPU's dispatched inputs
    xp = to_host(d["x_perm"][torch.from_numpy(rows).long().cuda()])
    sub_indptr = ref["m_indptr"]
    full_xperm = np.zeros((R, H), np.uint16)  # only the sampled rows are read by the oracle
    full_xperm[rows] = xp
    rh, _, ry = oracle.grouped_swiglu_rows(full_xperm, sub_indptr, inp["wgu"], inp["wd"], to_host(d["w_perm"]), rows)
    ridx = torch.from_numpy(rows).long().cuda()
    assert_close(bf16_to_f64(to_host(h[ridx])), bf16_to_f64(rh), f"{name} h rows")
    assert_close(bf16_to_f64(to_host(y_perm[ridx])), bf16_to_f64(ry), f"{name} y rows")

    # whole-layer output and token gradients of sampled tokens
    tidx = torch.from_numpy(toks).long().cuda()
    rY = oracle.forward_tokens(inp["x"], inp["wgu"], inp["wd"], rids, rw, toks=toks)
    assert_close(bf16_to_f64(to_host(Y[tidx])), bf16_to_f64(rY), f"{name} Y")
    rdx, rdl = oracle.backward_tokens(inp["x"], inp["dy"], inp["wgu"], inp["wd"], rids, rw, toks=toks)
    assert_close(bf16_to_f64(to_host(dx[tidx])), bf16_to_f64(rdx), f"{name} dX")
    dl_h = to_host(dl[tidx])
    assert_close(dl_h, rdl, f"{name} d_logits")
    assert np.all(dl_h[rdl == 0] == 0)

    # weight gradients of sampled experts
    exps = _sample_experts(ref["counts"])
    rdwgu, rdwd = oracle.backward_dw(inp["x"], inp["dy"], inp["wgu"], inp["wd"], rids, rw, experts=exps)
    eidx = torch.from_numpy(exps).long().cuda()
    assert_close(bf16_to_f64(to_host(dwgu[eidx])), bf16_to_f64(rdwgu), f"{name} dW_gate_up", per_expert=True)
    assert_close(bf16_to_f64(to_host(dwd[eidx])), bf16_to_f64(rdwd), f"{name} dW_down", per_expert=True)
    empty = np.nonzero(ref["counts"] == 0)[0][:4]
    if empty.size:
        e2 = torch.from_numpy(empty).long().cuda()
        assert torch.count_nonzero(dwgu[e2]) == 0 and torch.count_nonzero(dwd[e2]) == 0
