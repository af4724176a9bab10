"""Pins for the oracle's router projection (logits = x Wr^T + b) and its backward, CPU only.

The pages leave the router to the host framework (LightMoE README, "MoE training": routing
policy is the framework's responsibility); its plainest form is one bias-optional linear layer.
Nothing below takes an expected value from the oracle:
- the forward against an fp64 matmul within the fp32 recursive-summation bound;
- the backward against fp64 autograd of <d_logits, x Wr^T + b> for a dense d_logits;
- the whole layer with the router inside the graph (x -> logits -> top-k softmax -> experts)
  against fp64 autograd: the layer's dX plus the router's dX is the total input gradient;
- closed forms and degenerate cases (k = 1 gives no router gradient at all).
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from tests.helpers import bf16_to_f64, rel_errors, rel_errors_per_expert

# bf16 outputs against exact fp64: one rounding of 2^-9 relative (at most one ulp apart near a
# rounding midpoint, where the fp32 sum and the exact value fall on either side).
ONE_ULP = 2.0 ** -7

SHAPES = [(64, 320, 37), (33, 128, 8), (1, 64, 1)]


def _inputs(T, H, E, seed=3):
    x = synthetic.normal_bf16((T, H), seed, synthetic.STREAM_X, 1.0)
    wr = synthetic.normal_bf16((E, H), seed, synthetic.STREAM_WR, 0.3)
    rng = np.random.default_rng(seed)
    bias = rng.normal(0.0, 0.5, E).astype(np.float32)
    return x, wr, bias


@pytest.mark.parametrize("T,H,E", SHAPES)
@pytest.mark.parametrize("with_bias", [True, False])
def test_logits_match_fp64_within_summation_bound(T, H, E, with_bias):
    x, wr, bias = _inputs(T, H, E)
    b = bias if with_bias else None
    got = oracle.router_logits(x, wr, b).astype(np.float64)
    X, W = bf16_to_f64(x), bf16_to_f64(wr)
    exact = X @ W.T + (bias.astype(np.float64) if with_bias else 0.0)
    # recursive float summation of H exact products, then one add: |err| <= (H+1) u sum|terms|
    mag = np.abs(X) @ np.abs(W).T + (np.abs(bias.astype(np.float64)) if with_bias else 0.0)
    bound = (H + 1) * 2.0 ** -24 * mag + 1e-30
    assert np.all(np.abs(got - exact) <= bound)


def test_logits_equal_the_input_recipe_sum():
    """The generator's route_topk input (a double sum rounded once) agrees within the float bound."""
    wl = synthetic.Workload("zipf_T40_H256_I64_E16_k4", 40, 256, 64, 16, 4, zipf_s=1.2)
    inp = synthetic.make_inputs(wl, want=("x", "logits", "wr"))
    got = oracle.router_logits(inp["x"], inp["wr"], inp["bias"]).astype(np.float64)
    mag = np.abs(bf16_to_f64(inp["x"])) @ np.abs(bf16_to_f64(inp["wr"])).T + np.abs(inp["bias"])
    assert np.all(np.abs(got - inp["logits"]) <= (wl.H + 2) * 2.0 ** -24 * mag + 1e-30)


def test_closed_form_values():
    # x = [1, 2]; Wr rows [1, 1] and [2, -1]; b = [0.5, -1] -> logits [3.5, -1]
    one, two, mone = 0x3F80, 0x4000, 0xBF80
    x = np.array([[one, two]], np.uint16)
    wr = np.array([[one, one], [two, mone]], np.uint16)
    np.testing.assert_array_equal(oracle.router_logits(x, wr, np.array([0.5, -1.0], np.float32)), [[3.5, -1.0]])
    # backward with d_logits = [1, -2]: dX = dx_in + [1 - 4, 1 + 2] = [0.5 - 3, 3]; dWr = [[1, 2], [-2, -4]]
    dl = np.array([[1.0, -2.0]], np.float32)
    dx_in = np.array([[0x3F00, 0x0000]], np.uint16)  # [0.5, 0]
    dx, dwr, db = oracle.router_backward(dl, x, wr, dx_in)
    np.testing.assert_array_equal(bf16_to_f64(dx), [[-2.5, 3.0]])
    np.testing.assert_array_equal(bf16_to_f64(dwr), [[1.0, 2.0], [-2.0, -4.0]])
    np.testing.assert_array_equal(db, [1.0, -2.0])


@pytest.mark.parametrize("T,H,E", SHAPES)
@pytest.mark.parametrize("with_dx_in", [True, False])
def test_backward_matches_fp64_autograd_dense(T, H, E, with_dx_in):
    x, wr, bias = _inputs(T, H, E)
    rng = np.random.default_rng(11)
    dl = rng.normal(0.0, 1.0, (T, E)).astype(np.float32)  # dense: every entry counts
    dx_in = synthetic.normal_bf16((T, H), 5, synthetic.STREAM_DY, 0.1) if with_dx_in else None
    dx, dwr, db = oracle.router_backward(dl, x, wr, dx_in)
    X = torch.tensor(bf16_to_f64(x), requires_grad=True)
    W = torch.tensor(bf16_to_f64(wr), requires_grad=True)
    B = torch.tensor(bias.astype(np.float64), requires_grad=True)
    (torch.tensor(dl.astype(np.float64)) * (X @ W.T + B)).sum().backward()
    ref_dx = X.grad.numpy() + (bf16_to_f64(dx_in) if with_dx_in else 0.0)
    for name, got, ref in (("dX", bf16_to_f64(dx), ref_dx), ("dWr", bf16_to_f64(dwr), W.grad.numpy())):
        mx, mn = rel_errors(got, ref)
        assert mx <= ONE_ULP and mn <= 2.0 ** -9, (name, mx, mn)
    np.testing.assert_allclose(db, B.grad.numpy(), rtol=T * 2.0 ** -23, atol=1e-30)


def test_backward_subsets_equal_the_full_call():
    x, wr, _ = _inputs(40, 128, 9)
    dl = np.random.default_rng(2).normal(0.0, 1.0, (40, 9)).astype(np.float32)
    dx, dwr, db = oracle.router_backward(dl, x, wr)
    toks, exps = np.array([39, 0, 7], np.int32), np.array([8, 2], np.int32)
    dx_s, dwr_s, db_s = oracle.router_backward(dl, x, wr, toks=toks, experts=exps)
    np.testing.assert_array_equal(dx_s, dx[toks])
    np.testing.assert_array_equal(dwr_s, dwr[exps])
    np.testing.assert_array_equal(db_s, db[exps])


LAYERS = [
    synthetic.Workload("tiny_T64_H128_I64_E8_k2", 64, 128, 64, 8, 2, router_std=0.2),
    synthetic.Workload("zipf_T96_H128_I64_E16_k4", 96, 128, 64, 16, 4, zipf_s=1.2, router_std=0.2),
]


@pytest.mark.parametrize("wl", LAYERS, ids=lambda w: w.name)
def test_layer_with_router_matches_fp64_autograd(wl):
    """x -> logits = x Wr^T + b -> top-k softmax -> experts -> Y, loss <dY, Y>, all in fp64 autograd;
    the oracle's path: router_logits -> route_topk -> backward_tokens (layer dX, d_logits) ->
    router_backward (adds the router's dX, gives dWr, dbias)."""
    inp = synthetic.make_inputs(wl, want=("x", "wr", "wgu", "wd", "dy"))
    logits = oracle.router_logits(inp["x"], inp["wr"], inp["bias"])
    ids, w = oracle.route_topk(logits, wl.k)
    dx_layer, dl = oracle.backward_tokens(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w)
    dx, dwr, db = oracle.router_backward(dl, inp["x"], inp["wr"], dx_layer)

    # x enters twice (router input Xr, expert input Xe); the total input gradient is the sum
    Xr = torch.tensor(bf16_to_f64(inp["x"]), requires_grad=True)
    Xe = torch.tensor(bf16_to_f64(inp["x"]), requires_grad=True)
    Wr = torch.tensor(bf16_to_f64(inp["wr"]), requires_grad=True)
    b = torch.zeros(wl.E, dtype=torch.float64) if inp["bias"] is None else torch.tensor(inp["bias"].astype(np.float64))
    b.requires_grad_(True)
    Wgu, Wd = torch.tensor(bf16_to_f64(inp["wgu"])), torch.tensor(bf16_to_f64(inp["wd"]))
    lg = Xr @ Wr.T + b
    # the selection is piecewise constant in the logits: fixed to the oracle's, the weights are
    # the softmax over it of the differentiable logits
    mask = torch.zeros((wl.T, wl.E), dtype=torch.bool)
    mask[torch.arange(wl.T)[:, None], torch.tensor(ids, dtype=torch.long)] = True
    G = torch.softmax(lg.masked_fill(~mask, float("-inf")), dim=1)
    gu = torch.einsum("th,enh->ten", Xe, Wgu)
    a = torch.nn.functional.silu(gu[..., : wl.I]) * gu[..., wl.I:]
    Y = torch.einsum("te,tec->tc", G, torch.einsum("ten,ecn->tec", a, Wd))
    ((Y * torch.tensor(bf16_to_f64(inp["dy"]))).sum()).backward()
    total_dx = Xe.grad.numpy() + Xr.grad.numpy()
    mx, mn = rel_errors(bf16_to_f64(dx), total_dx)
    assert mx <= 1.5e-2 and mn <= 3e-3, ("dX", mx, mn)
    mx, mn = rel_errors_per_expert(bf16_to_f64(dwr)[:, None, :], Wr.grad.numpy()[:, None, :])
    assert mx <= 1.5e-2 and mn <= 3e-3, ("dWr", mx, mn)
    # dbias is a sum of d_logits, which carry the bf16 rounding of h (the layer's own bar)
    mx, mn = rel_errors(db, b.grad.numpy())
    assert mx <= 1.5e-2 and mn <= 3e-3, ("dbias", mx, mn)
    # the router's share is not negligible in this test (so a dropped router term fails it)
    assert np.abs(Xr.grad.numpy()).sum() > 0.05 * np.abs(Xe.grad.numpy()).sum()


def test_top1_routing_gives_no_router_gradient():
    """k = 1: the renormalised weight is 1 for every logit, so d_logits = 0, dWr = 0, dbias = 0 and
    the router leaves dX unchanged, exactly."""
    wl = synthetic.Workload("top1_T50_H64_I64_E6_k1", 50, 64, 64, 6, 1, router_std=0.3)
    inp = synthetic.make_inputs(wl, want=("x", "wr", "wgu", "wd", "dy"))
    ids, w = oracle.route_topk(oracle.router_logits(inp["x"], inp["wr"], None), 1)
    dx_layer, dl = oracle.backward_tokens(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w)
    assert np.all(dl == 0)
    dx, dwr, db = oracle.router_backward(dl, inp["x"], inp["wr"], dx_layer)
    np.testing.assert_array_equal(dx, dx_layer)
    assert np.all(bf16_to_f64(dwr) == 0) and np.all(db == 0)
