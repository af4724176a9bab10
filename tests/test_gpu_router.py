"""GPU parity of the router projection (logits = x Wr^T + b) and its backward against the oracle.

The pages leave the router to the host framework (LightMoE README, "MoE training"); this library's
router is one bias-optional linear layer.  Bars:
- logits (fp32): within the fp32 summation bound of the exact sum, |err| <= 4 (H + 1) 2^-24 sum|x w|
  (the tensor cores add in another order than a sequential loop, so not bit for bit);
- routing: ids bit-exact given the GPU's logits (the oracle's top-k of the same float32 bytes),
  weights within 2e-6 relative (the device exp and the host exp differ by an ulp or two);
- dX, dWr (bf16): max_rel 2e-2 / mean_rel 1e-2 (dWr per expert); dbias (fp32): 1e-4.
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

# (T, H, E, bias): ragged M tails, E below / above one 256-column tile, E a multiple of 32 (TMA
# stores) or not (element stores), and the bench workload's router shape
LOGIT_SHAPES = [(256, 256, 8, True), (300, 320, 37, False), (513, 256, 512, True), (200, 128, 600, True),
                (1000, 2048, 256, False), (1, 64, 1, True)]


def _router_inputs(T, H, E, seed=7):
    x = synthetic.normal_bf16((T, H), seed, synthetic.STREAM_X, 1.0)
    wr = synthetic.normal_bf16((E, H), seed, synthetic.STREAM_WR, 0.05)
    bias = np.random.default_rng(seed).normal(0.0, 0.5, E).astype(np.float32)
    return x, wr, bias


def _check_logits(got, x, wr, bias):
    X, W = bf16_to_f64(x), bf16_to_f64(wr)
    exact = X @ W.T + (0.0 if bias is None else bias.astype(np.float64))
    mag = np.abs(X) @ np.abs(W).T + (0.0 if bias is None else np.abs(bias.astype(np.float64)))
    bound = 4 * (X.shape[1] + 1) * 2.0 ** -24 * mag + 1e-30
    err = np.abs(got.astype(np.float64) - exact)
    assert np.all(err <= bound), float((err / bound).max())


@pytest.mark.parametrize("T,H,E,with_bias", LOGIT_SHAPES)
def test_logits_parity(T, H, E, with_bias):
    x, wr, bias = _router_inputs(T, H, E)
    b = bias if with_bias else None
    got = to_host(moe.router_logits(to_dev(x), to_dev(wr), None if b is None else to_dev(b)))
    assert moe.device_error() == 0
    _check_logits(got, x, wr, b)
    # and against the oracle's sequential fp32 sum: both sit within the bound of the exact value
    ref = oracle.router_logits(x, wr, b).astype(np.float64)
    X, Wm = np.abs(bf16_to_f64(x)), np.abs(bf16_to_f64(wr))
    mag = X @ Wm.T + (0.0 if b is None else np.abs(b.astype(np.float64)))
    assert np.all(np.abs(got - ref) <= 5 * (H + 1) * 2.0 ** -24 * mag + 1e-30)


def test_zero_tokens_launch_nothing():
    x = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    wr = to_dev(synthetic.normal_bf16((8, 128), 0, synthetic.STREAM_WR, 0.1))
    assert moe.router_logits(x, wr).shape == (0, 8)
    assert moe.device_error() == 0


W = synthetic.Workload
LAYERS = [
    W("tiny_T256_H256_I128_E8_k2", 256, 256, 128, 8, 2, router_std=0.1),
    W("many_T300_H128_I64_E37_k5", 300, 128, 64, 37, 5, router_std=0.1),
    W("zipf_T512_H256_I128_E16_k4", 512, 256, 128, 16, 4, zipf_s=1.2, router_std=0.3),  # empty experts
]


def _gpu_layer(wl, inp, logits_dev):
    """GPU: route the GPU logits, dispatch, expert MLP, combine, backward, router backward."""
    ids, w = moe.route_topk(logits_dev, wl.k)
    x = to_dev(inp["x"])
    wgu, wd, wr = to_dev(inp["wgu"]), to_dev(inp["wd"]), to_dev(inp["wr"])
    d = moe.dispatch(ids, w, x, wl.E)
    h, gu, y_perm = moe.grouped_swiglu_fwd(d["x_perm"], d["m_indptr"], wgu, wd, d["w_perm"])
    Y = moe.combine(y_perm, d["slot_to_row"], wl.T, wl.k)
    dx, _, _, dl = moe.bwd_dx_dw(to_dev(inp["dy"]), d["x_perm"], h, gu, ids, w, d["m_indptr"], d["row_to_slot"],
                                 d["slot_to_row"], d["w_perm"], wgu, wd)
    dx_layer = dx.clone()
    dwr, db = moe.router_bwd(dl, ids, d["m_indptr"], d["row_to_slot"], x, wr, dx)
    return dict(ids=ids, w=w, d=d, Y=Y, dx_layer=dx_layer, dx=dx, dl=dl, dwr=dwr, db=db)


@pytest.mark.parametrize("wl", LAYERS, ids=lambda w: w.name)
def test_router_backward_parity_on_shared_inputs(wl):
    """router_bwd alone: both sides take the oracle's d_logits, routing and layer dX."""
    inp = synthetic.make_inputs(wl, want=("x", "wr", "wgu", "wd", "dy"))
    logits = oracle.router_logits(inp["x"], inp["wr"], inp["bias"])
    ids, w = oracle.route_topk(logits, wl.k)
    ref_d = oracle.dispatch(ids, w, None, wl.E)
    dx_layer, dl = oracle.backward_tokens(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w)
    rdx, rdwr, rdb = oracle.router_backward(dl, inp["x"], inp["wr"], dx_layer)
    dx = to_dev(dx_layer)
    dwr, db = moe.router_bwd(to_dev(dl), to_dev(ids), to_dev(ref_d["m_indptr"]), to_dev(ref_d["row_to_slot"]),
                             to_dev(inp["x"]), to_dev(inp["wr"]), dx)
    assert moe.device_error() == 0
    assert_close(bf16_to_f64(to_host(dx)), bf16_to_f64(rdx), "dX (layer + router)")
    assert_close(bf16_to_f64(to_host(dwr))[:, None, :], bf16_to_f64(rdwr)[:, None, :], "dWr", per_expert=True)
    assert_close(to_host(db), rdb, "dbias", max_rel=1e-4, mean_rel=1e-5)
    counts = np.bincount(ids.ravel(), minlength=wl.E)
    assert np.all(to_host(dwr)[counts == 0] == 0) and np.all(to_host(db)[counts == 0] == 0)
    # the router term alone (dx_in = 0) also meets the bar
    dx0 = torch.zeros_like(dx)
    moe.router_bwd(to_dev(dl), to_dev(ids), to_dev(ref_d["m_indptr"]), to_dev(ref_d["row_to_slot"]),
                   to_dev(inp["x"]), to_dev(inp["wr"]), dx0)
    r0, _, _ = oracle.router_backward(dl, inp["x"], inp["wr"], None, experts=np.zeros(0, np.int32))
    assert_close(bf16_to_f64(to_host(dx0)), bf16_to_f64(r0), "dX (router term alone)")


@pytest.mark.parametrize("wl", LAYERS, ids=lambda w: w.name)
def test_layer_with_router_parity(wl):
    """The whole GPU path from x: router logits -> top-k -> layer -> backward -> router backward,
    against the oracle on the GPU's logits (routing is bit-exact given those logits)."""
    inp = synthetic.make_inputs(wl, want=("x", "wr", "wgu", "wd", "dy"))
    bias = None if inp["bias"] is None else to_dev(inp["bias"])
    lg = moe.router_logits(to_dev(inp["x"]), to_dev(inp["wr"]), bias)
    g = _gpu_layer(wl, inp, lg)
    assert moe.device_error() == 0
    lg_h = to_host(lg)
    _check_logits(lg_h, inp["x"], inp["wr"], inp["bias"])
    ids, w = oracle.route_topk(lg_h, wl.k)
    np.testing.assert_array_equal(to_host(g["ids"]), ids)
    np.testing.assert_allclose(to_host(g["w"]), w, rtol=2e-6, atol=1e-8)  # expf vs std::exp: an ulp or two
    Y = oracle.forward_tokens(inp["x"], inp["wgu"], inp["wd"], ids, w)
    assert_close(bf16_to_f64(to_host(g["Y"])), bf16_to_f64(Y), "Y")
    dx_layer, dl = oracle.backward_tokens(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w)
    rdx, rdwr, rdb = oracle.router_backward(dl, inp["x"], inp["wr"], dx_layer)
    assert_close(bf16_to_f64(to_host(g["dx"])), bf16_to_f64(rdx), "dX")
    assert_close(bf16_to_f64(to_host(g["dwr"]))[:, None, :], bf16_to_f64(rdwr)[:, None, :], "dWr", per_expert=True)
    assert_close(to_host(g["db"]), rdb, "dbias", max_rel=2e-2, mean_rel=1e-2)  # inherits d_logits' bf16 bar


def test_top1_leaves_dx_unchanged():
    """k = 1: d_logits = 0, so the router adds exactly nothing and its gradients are exact zeros."""
    wl = W("top1_T300_H128_I64_E6_k1", 300, 128, 64, 6, 1, router_std=0.3)
    inp = synthetic.make_inputs(wl, want=("x", "wr", "wgu", "wd", "dy"))
    g = _gpu_layer(wl, inp, moe.router_logits(to_dev(inp["x"]), to_dev(inp["wr"])))
    assert moe.device_error() == 0
    assert torch.count_nonzero(g["dl"]) == 0
    assert torch.equal(g["dx"], g["dx_layer"])
    assert torch.count_nonzero(g["dwr"].float()) == 0 and torch.count_nonzero(g["db"]) == 0


def test_bad_expert_id_is_flagged_and_leaves_the_token():
    wl = W("flag_T64_H128_I64_E8_k2", 64, 128, 64, 8, 2)
    x, wr, _ = _router_inputs(wl.T, wl.H, wl.E)
    ids = np.tile(np.array([[0, 1]], np.int32), (wl.T, 1))
    ids[5, 1] = 99  # out of range
    d = oracle.dispatch(np.tile(np.array([[0, 1]], np.int32), (wl.T, 1)), None, None, wl.E)
    dl = np.zeros((wl.T, wl.E), np.float32)
    dl[:, 0], dl[:, 1] = 0.25, -0.25
    dx = torch.zeros((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    moe.router_bwd(to_dev(dl), to_dev(ids), to_dev(d["m_indptr"]), to_dev(d["row_to_slot"]), to_dev(x), to_dev(wr),
                   dx)
    assert moe.device_error() == moe_deverr("BAD_EXPERT_ID")
    assert torch.count_nonzero(dx[5]) == 0 and torch.count_nonzero(dx[4]) > 0


def moe_deverr(name):
    return {v: k for k, v in moe.DEVERR.items()}[name]


# Full size: the router shapes of the bench workload (T=8192, H=2048, E=256, k=8) and of the
# Zipf-skewed 4096/1024 workload (T=8192, H=4096, E=512, k=10, with its load-skew bias).
FULL = ["fwd_T8192_H2048_I512_E256_k8", "fwd_zipf_T8192_H4096_I1024_E512_k10"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_router(name):
    wl = synthetic.WORKLOADS[name]
    inp = synthetic.make_inputs(wl, want=("x", "wr"))
    x, wr = to_dev(inp["x"]), to_dev(inp["wr"])
    bias = None if inp["bias"] is None else to_dev(inp["bias"])
    lg = moe.router_logits(x, wr, bias)
    ids, w = moe.route_topk(lg, wl.k)
    d = moe.dispatch(ids, w, None, wl.E)
    assert moe.device_error() == 0
    lg_h, ids_h = to_host(lg), to_host(ids)
    _check_logits(lg_h, inp["x"], inp["wr"], inp["bias"])  # every logit
    rids, rw = oracle.route_topk(lg_h, wl.k)
    np.testing.assert_array_equal(ids_h, rids)  # routing bit-exact given the GPU's logits
    # a d_logits with the layer's sparsity: values at the selected entries, zero elsewhere
    rng = np.random.default_rng(1)
    dl = np.zeros((wl.T, wl.E), np.float32)
    np.put_along_axis(dl, ids_h.astype(np.int64), rng.normal(0.0, 0.05, ids_h.shape).astype(np.float32), axis=1)
    dx_in = synthetic.normal_bf16((wl.T, wl.H), 3, synthetic.STREAM_DY, 1.0)
    dx = to_dev(dx_in)
    dwr, db = moe.router_bwd(to_dev(dl), ids, d["m_indptr"], d["row_to_slot"], x, wr, dx)
    assert moe.device_error() == 0
    toks = np.unique(np.random.default_rng(2).integers(0, wl.T, 48)).astype(np.int32)
    counts = np.bincount(ids_h.ravel(), minlength=wl.E)
    nz = np.nonzero(counts)[0]
    order = nz[np.argsort(counts[nz], kind="stable")]
    exps = np.unique(np.array([order[0], order[len(order) // 2], order[-1]], np.int32))
    rdx, rdwr, rdb = oracle.router_backward(dl, inp["x"], inp["wr"], dx_in, toks=toks, experts=exps)
    assert_close(bf16_to_f64(to_host(dx)[toks]), bf16_to_f64(rdx), "dX (sampled tokens)")
    assert_close(bf16_to_f64(to_host(dwr)[exps])[:, None, :], bf16_to_f64(rdwr)[:, None, :], "dWr (sampled experts)",
                 per_expert=True)
    assert_close(to_host(db), dl.astype(np.float64).sum(0), "dbias", max_rel=1e-4, mean_rel=1e-5)
    empty = counts == 0
    assert np.all(to_host(dwr)[empty] == 0) and np.all(to_host(db)[empty] == 0)
