"""Full-size parity on every workload shape, in the launch configuration the benchmark uses
(dispatch writes x_perm; the expert GEMMs read expert-major tiles).

Routing ids, counts, m_indptr and both permutations are compared whole and must
be bit-exact.  Float outputs are compared on samples the oracle computes one by
one: the layer output Y, dX and d_logits of sampled tokens, h / y of sampled
rows, and the weight gradients of sampled experts (the lightest non-empty one,
a median one and the heaviest one up to a row budget; in the composed check also
the heaviest one of all, whose K loop is the longest the weight-gradient GEMMs
run).  Besides the five workloads, the training shape runs at 1024 and 16384
tokens (the ends of the pages' tokens-per-rank sweep).

Two backward checks:
* isolated: the backward entry point gets the same saved forward state on both
  sides (the rows that feed the sampled outputs come from the oracle's forward);
  every output meets the bar.
* composed: GPU forward then GPU backward.  h is stored in bf16 by both sides,
  and where silu(g)*u lies next to a bf16 rounding midpoint the two fp32
  accumulation orders round it to neighbouring values; where g or u lies near
  zero, those orders move g or u themselves by a relative amount large enough to
  shift h by several ulps.  Every h that enters the dW_down bound is checked:
  within one bf16 ulp of the oracle's, or within one ulp plus the activation's
  sensitivity times the fp32 summation bound of g and u (_assert_h_explained).
  dW_down sums h over rows, so its bound adds the exact propagation of those
  differences, sum_r |w_r dY[r,c]| * |h_gpu - h_oracle|[r,n].
"""
import numpy as np
import pytest
import torch

import mixture_experts_routed_router_gb300 as moe
import oracle
import synthetic
from tests.gpu_util import dw_fp16, to_dev, to_host
from tests.helpers import MAX_REL_TOL, MEAN_REL_TOL, assert_close, bf16_to_f64, rel_errors, swiglu_factors, off_selection

pytestmark = pytest.mark.gpu

N_TOKENS = 24
ROW_BUDGET = 1200  # rows of the sampled experts whose dW the oracle recomputes
# the training shape at the ends of the tokens-per-rank sweep
SWEEP = ["train_T1024_H2048_I768_E128_k8", "train_T16384_H2048_I768_E128_k8"]


def _rows_of(exps, m_indptr):
    return np.concatenate([np.arange(m_indptr[e], m_indptr[e + 1]) for e in exps]).astype(np.int32)


def _bf16_ulps(a, b):
    """Distance in bf16 units in the last place between arrays of bf16 bit patterns."""
    def ordered(v):
        v = v.astype(np.int32)
        return np.where(v & 0x8000, -(v & 0x7FFF), v)
    return np.abs(ordered(a) - ordered(b))


# Two fp32 sums of the same H products in different orders differ by at most this many multiples of
# 2^-24 sqrt(H) ||x o w||_2 (x o w the products).  The oracle's sequential sum stays within 3 of the
# exact value on the Zipf workload's heaviest expert; 16 leaves room for the tensor cores' order.
SUM_ORDER_KAPPA = 16.0


def _assert_h_explained(name, e, x_rows, wgu_e, h_gpu, h_ref, gu_ref):
    """h_gpu within one bf16 ulp of the oracle's h, or within one ulp plus |dh/dg| dg + |dh/du| du,
    where dg, du bound the difference between two fp32 summation orders of g and u.  A wrong h
    (a wrong weight row, a dropped term) is far outside either bound."""
    ulps = _bf16_ulps(h_gpu, h_ref)
    if ulps.max() <= 1:
        return
    X, W = bf16_to_f64(x_rows), bf16_to_f64(wgu_e)
    I = W.shape[0] // 2
    unit = SUM_ORDER_KAPPA * 2.0 ** -24 * np.sqrt(X.shape[1])
    X2, W2 = X * X, W * W
    dg, du = unit * np.sqrt(X2 @ W2[:I].T), unit * np.sqrt(X2 @ W2[I:].T)
    f = swiglu_factors(gu_ref).astype(np.float64)
    ho, hg = bf16_to_f64(h_ref), bf16_to_f64(h_gpu)
    ulp = np.spacing(np.abs(ho).astype(np.float32)).astype(np.float64) * 65536.0
    allow = ulp + np.abs(f[:, :I]) * dg + np.abs(f[:, I:]) * du
    bad = (ulps > 1) & (np.abs(hg - ho) > allow)
    assert not bad.any(), (f"{name} expert {e}: {int(bad.sum())} h values differ from the oracle's beyond one "
                           f"ulp and the fp32 summation bound (worst {ulps[bad].max()} ulps)")


def _assert_dwd_with_h_allowance(name, wl, got, ref_bits, exps, disp, inp, w_ref, h_gpu):
    """dW_down of sampled experts within the bar plus the propagated h differences."""
    rows = _rows_of(exps, disp["m_indptr"])
    xp = np.zeros((wl.R, wl.H), np.uint16)
    xp[rows] = inp["x"][disp["row_to_slot"][rows] // wl.k]
    hq, gq, _ = oracle.grouped_swiglu_rows(xp, disp["m_indptr"], inp["wgu"], inp["wd"],
                                           w_ref.ravel()[disp["row_to_slot"]], rows)
    hq_oracle, gu_oracle = dict(zip(rows.tolist(), hq)), dict(zip(rows.tolist(), gq))
    dy = bf16_to_f64(inp["dy"])
    w_flat = w_ref.ravel()
    worst = 0.0
    for i, e in enumerate(exps):
        rows = np.arange(disp["m_indptr"][e], disp["m_indptr"][e + 1])
        slots = disp["row_to_slot"][rows]
        h_ref = np.stack([hq_oracle[r] for r in rows.tolist()])
        _assert_h_explained(name, e, xp[rows], inp["wgu"][e], h_gpu[rows], h_ref,
                            np.stack([gu_oracle[r] for r in rows.tolist()]))
        dh = np.abs(bf16_to_f64(h_gpu[rows]) - bf16_to_f64(h_ref))
        allow = (np.abs(w_flat[slots])[:, None] * np.abs(dy[slots // wl.k])).T @ dh  # [H, I]
        g, o = bf16_to_f64(got[i]), bf16_to_f64(ref_bits[i])
        rms = float(np.sqrt(np.mean(o * o)))
        excess = np.abs(g - o) - allow
        ratio = float(np.max(excess / np.maximum(np.abs(o), rms)))
        worst = max(worst, ratio)
    _, mean_rel = rel_errors(bf16_to_f64(got), bf16_to_f64(ref_bits))
    assert worst <= MAX_REL_TOL and mean_rel <= MEAN_REL_TOL, \
        f"{name} dW_down: max_rel beyond the h-difference allowance {worst:.3e}, mean_rel {mean_rel:.3e}"


def _sample_experts(counts, heaviest=False):
    nz = np.nonzero(counts)[0]
    order = nz[np.argsort(counts[nz], kind="stable")]
    picks = [order[0], order[len(order) // 2]]
    for e in order[::-1]:
        if counts[e] <= ROW_BUDGET:
            picks.append(e)
            break
    if heaviest:
        picks.append(order[-1])
    return np.unique(np.array(picks, dtype=np.int32))


@pytest.mark.parametrize("name", list(synthetic.WORKLOADS) + SWEEP)
def test_full_size_sampled_parity(name):
    wl = synthetic.workload(name)
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

    # expert MLP rows (h, y): each row's input is its token's x (the dispatch above is bit-exact)
    sub_indptr = ref["m_indptr"]
    full_xperm = np.zeros((R, H), np.uint16)  # only the sampled rows are read by the oracle
    full_xperm[rows] = inp["x"][ref["row_to_slot"][rows] // k]
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
    assert np.all(dl_h[off_selection(rids[toks], E)] == 0)

    # weight gradients of sampled experts, the heaviest one included
    exps = _sample_experts(ref["counts"], heaviest=True)
    rdwgu, rdwd = oracle.backward_dw(inp["x"], inp["dy"], inp["wgu"], inp["wd"], rids, rw, experts=exps)
    eidx = torch.from_numpy(exps).long().cuda()
    assert_close(bf16_to_f64(to_host(dwgu[eidx])), bf16_to_f64(rdwgu), f"{name} dW_gate_up", per_expert=True)
    _assert_dwd_with_h_allowance(name, wl, to_host(dwd[eidx]), rdwd, exps, ref, inp, rw, to_host(h))
    empty = np.nonzero(ref["counts"] == 0)[0][:4]
    if empty.size:
        e2 = torch.from_numpy(empty).long().cuda()
        assert torch.count_nonzero(dwgu[e2]) == 0 and torch.count_nonzero(dwd[e2]) == 0


@pytest.mark.parametrize("name", list(synthetic.WORKLOADS))
def test_full_size_backward_isolated(name):
    """The backward entry point on a saved forward state that both sides share."""
    wl = synthetic.WORKLOADS[name]
    inp = synthetic.make_inputs(wl, seed=0)
    T, H, I, E, k, R = wl.T, wl.H, wl.I, wl.E, wl.k, wl.R
    logits, x, dy = to_dev(inp["logits"]), to_dev(inp["x"]), to_dev(inp["dy"])
    wgu, wd = to_dev(inp["wgu"]), to_dev(inp["wd"])
    ids, w = moe.route_topk(logits, k)
    d = moe.dispatch(ids, w, x, E)
    h, gu, _ = moe.grouped_swiglu_fwd(d["x_perm"], d["m_indptr"], wgu, wd, d["w_perm"])
    rids, rw = oracle.route_topk(inp["logits"], k)
    ref = oracle.dispatch(rids, rw, None, E)
    np.testing.assert_array_equal(to_host(d["row_to_slot"]), ref["row_to_slot"])

    rng = np.random.default_rng(4321)
    toks = np.sort(rng.choice(T, size=min(N_TOKENS, T), replace=False)).astype(np.int32)
    exps = _sample_experts(ref["counts"])
    rows = np.union1d(_rows_of(exps, ref["m_indptr"]), ref["slot_to_row"].reshape(T, k)[toks].ravel()).astype(np.int32)
    # the saved state of these rows comes from the oracle's forward (the rest cannot reach the checked outputs)
    xp = np.zeros((R, H), np.uint16)
    xp[rows] = inp["x"][ref["row_to_slot"][rows] // k]
    w_perm_ref = rw.ravel()[ref["row_to_slot"]]
    rh, rgu, _ = oracle.grouped_swiglu_rows(xp, ref["m_indptr"], inp["wgu"], inp["wd"], w_perm_ref, rows)
    ridx = torch.from_numpy(rows).long().cuda()
    h[ridx] = to_dev(rh)
    gu[ridx] = torch.from_numpy(swiglu_factors(rgu)).cuda()
    w_perm = to_dev(w_perm_ref)
    dx, dwgu, dwd, dl = moe.bwd_dx_dw(dy, d["x_perm"], h, gu, ids, to_dev(rw), d["m_indptr"], d["row_to_slot"],
                                      d["slot_to_row"], w_perm, wgu, wd)
    assert moe.device_error() == 0
    tidx = torch.from_numpy(toks).long().cuda()
    rdx, rdl = oracle.backward_tokens(inp["x"], inp["dy"], inp["wgu"], inp["wd"], rids, rw, toks=toks)
    assert_close(bf16_to_f64(to_host(dx[tidx])), bf16_to_f64(rdx), f"{name} dX (isolated)")
    assert_close(to_host(dl[tidx]), rdl, f"{name} d_logits (isolated)")
    rdwgu, rdwd = oracle.backward_dw(inp["x"], inp["dy"], inp["wgu"], inp["wd"], rids, rw, experts=exps)
    eidx = torch.from_numpy(exps).long().cuda()
    assert_close(bf16_to_f64(to_host(dwgu[eidx])), bf16_to_f64(rdwgu), f"{name} dW_gate_up (isolated)", per_expert=True)
    assert_close(bf16_to_f64(to_host(dwd[eidx])), bf16_to_f64(rdwd), f"{name} dW_down (isolated)", per_expert=True)


def test_full_size_gathered_and_dispatched_inputs_agree_bitwise():
    """On the benchmark's workload, the x_perm entry points give the same bits as the gathered ones."""
    wl = synthetic.WORKLOADS["fwd_T8192_H2048_I512_E256_k8"]
    inp = synthetic.make_inputs(wl, seed=0)
    k, E = wl.k, wl.E
    logits, x, dy = to_dev(inp["logits"]), to_dev(inp["x"]), to_dev(inp["dy"])
    wgu, wd = to_dev(inp["wgu"]), to_dev(inp["wd"])
    ids, w = moe.route_topk(logits, k)
    d = moe.dispatch(ids, w, x, E)
    ga = moe.grouped_swiglu_fwd_gather(x, d["row_to_slot"], k, d["m_indptr"], wgu, wd, d["w_perm"])
    pa = moe.grouped_swiglu_fwd(d["x_perm"], d["m_indptr"], wgu, wd, d["w_perm"])
    for u, v, name in zip(ga, pa, ("h", "gu", "y_perm")):
        assert torch.equal(u, v), name
    h, gu, _ = ga
    del pa
    common = (h, gu, ids, w, d["m_indptr"], d["row_to_slot"], d["slot_to_row"], d["w_perm"], wgu, wd)
    gb = moe.bwd_dx_dw_gather(dy, x, *common)
    with dw_fp16(False):  # the gathered backward takes the hi / lo weight-gradient operands
        pb = moe.bwd_dx_dw(dy, d["x_perm"], *common)
    for u, v, name in zip(gb, pb, ("dX", "dW_gate_up", "dW_down", "d_logits")):
        assert torch.equal(u, v), name
    assert moe.device_error() == 0
