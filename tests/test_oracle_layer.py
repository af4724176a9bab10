"""Pins for the oracle's expert MLP, combine, forward and backward, CPU only.

The expected values never come from the oracle: they come from an fp64 dense
evaluation with torch (every expert on every token, masked by the dense gate
matrix), torch.autograd on that dense form, central finite differences,
closed forms and degenerate cases.  The bars below are the bf16 rounding the
oracle performs by definition (h, y, Y and the gradients are stored bf16),
far below what a dropped term, a sign or an index error produces.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synthetic
from tests.helpers import (bf16_to_f64, dense_layer_fp64, dense_swiglu_mlp_fp64, rel_errors,
                           rel_errors_per_expert, topk_bruteforce)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_worked_example.json")

# Oracle vs exact fp64: the oracle rounds h, y, Y (and dX, dW) to bf16 (2^-9 relative each).
ORACLE_MAX_REL = 1.5e-2
ORACLE_MEAN_REL = 3e-3

TINY = synthetic.WORKLOADS["tiny_T256_H256_I128_E8_k2"]
RAGGED = synthetic.Workload("ragged_T50_H64_I64_E5_k3", 50, 64, 64, 5, 3)
ZIPF = synthetic.Workload("zipf_T96_H128_I64_E16_k4", 96, 128, 64, 16, 4, zipf_s=1.2, router_std=0.2)


def _case(wl):
    inp = synthetic.make_inputs(wl)
    ids, w = oracle.route_topk(inp["logits"], wl.k)
    return inp, ids, w


def _bits_of(t: torch.Tensor) -> np.ndarray:
    return synthetic.f32_to_bf16_bits(t.detach().numpy().astype(np.float32))


@pytest.mark.parametrize("wl", [TINY, RAGGED, ZIPF], ids=lambda w: w.name)
def test_forward_matches_fp64_dense(wl):
    inp, ids, w = _case(wl)
    np.testing.assert_array_equal(ids, topk_bruteforce(inp["logits"], wl.k))
    Y = oracle.forward_tokens(inp["x"], inp["wgu"], inp["wd"], ids, w)
    Yd, _ = dense_layer_fp64(inp["x"], inp["wgu"], inp["wd"], inp["logits"], ids)
    mx, mn = rel_errors(bf16_to_f64(Y), Yd.numpy())
    assert mx <= ORACLE_MAX_REL and mn <= ORACLE_MEAN_REL, (mx, mn)


@pytest.mark.parametrize("wl", [TINY, RAGGED, ZIPF], ids=lambda w: w.name)
def test_forward_is_dispatch_grouped_combine(wl):
    """The per-token forward equals dispatch -> grouped rows -> combine, bit for bit."""
    inp, ids, w = _case(wl)
    d = oracle.dispatch(ids, w, inp["x"], wl.E)
    rows = np.arange(wl.R, dtype=np.int32)
    h, gu, y = oracle.grouped_swiglu_rows(d["x_perm"], d["m_indptr"], inp["wgu"], inp["wd"], d["w_perm"], rows)
    Yc = oracle.combine(y, d["slot_to_row"], wl.T, wl.k)
    Yt = oracle.forward_tokens(inp["x"], inp["wgu"], inp["wd"], ids, w)
    np.testing.assert_array_equal(Yc, Yt)
    # intermediate h against fp64 (h = silu(g) * u before its bf16 rounding)
    e_of_row = np.searchsorted(d["m_indptr"], rows, side="right") - 1
    xr = torch.tensor(bf16_to_f64(d["x_perm"]))
    wgu = torch.tensor(bf16_to_f64(inp["wgu"]))[e_of_row]
    g = torch.einsum("rh,rnh->rn", xr, wgu[:, :wl.I])
    u = torch.einsum("rh,rnh->rn", xr, wgu[:, wl.I:])
    np.testing.assert_allclose(gu[:, :wl.I], g.numpy(), rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(gu[:, wl.I:], u.numpy(), rtol=1e-4, atol=1e-4)
    mx, mn = rel_errors(bf16_to_f64(h), (torch.nn.functional.silu(g) * u).numpy())
    assert mx <= 2 ** -8 and mn <= 2 ** -9


@pytest.mark.parametrize("wl", [TINY, RAGGED, ZIPF], ids=lambda w: w.name)
def test_backward_matches_fp64_autograd(wl):
    inp, ids, w = _case(wl)
    dX, dl = oracle.backward_tokens(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w)
    dwgu, dwd = oracle.backward_dw(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w)
    Yd, leaves = dense_layer_fp64(inp["x"], inp["wgu"], inp["wd"], inp["logits"], ids, requires_grad=True)
    dY = torch.tensor(bf16_to_f64(inp["dy"]))
    (Yd * dY).sum().backward()
    for name, got, ref, metric in (("dX", bf16_to_f64(dX), leaves["x"].grad, rel_errors),
                                   ("dW_gu", bf16_to_f64(dwgu), leaves["wgu"].grad, rel_errors_per_expert),
                                   ("dW_d", bf16_to_f64(dwd), leaves["wd"].grad, rel_errors_per_expert),
                                   ("d_logits", dl, leaves["logits"].grad, rel_errors)):
        mx, mn = metric(got, ref.numpy())
        assert mx <= ORACLE_MAX_REL and mn <= ORACLE_MEAN_REL, (name, mx, mn)
    # unselected logits get exactly zero gradient; each token's gradient sums to zero
    mask = np.zeros(dl.shape, bool)
    np.put_along_axis(mask, ids.astype(np.int64), True, axis=1)
    assert np.all(dl[~mask] == 0.0)
    scale = np.abs(dl).max(axis=1) + 1e-30
    assert np.all(np.abs(dl.astype(np.float64).sum(1)) <= 1e-5 * scale)


def test_router_gradient_by_central_differences():
    wl = RAGGED
    inp, ids, w = _case(wl)
    _, dl = oracle.backward_tokens(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w)
    dY = torch.tensor(bf16_to_f64(inp["dy"]))
    rng = np.random.default_rng(0)
    eps = 1e-5
    for t in rng.choice(wl.T, size=6, replace=False):
        for j in range(wl.k):
            e = ids[t, j]
            vals = []
            for sgn in (+1.0, -1.0):
                lg = inp["logits"].astype(np.float64).copy()
                lg[t, e] += sgn * eps
                Yd, _ = dense_layer_fp64(inp["x"], inp["wgu"], inp["wd"], lg, ids)
                vals.append(float((Yd * dY).sum()))
            fd = (vals[0] - vals[1]) / (2 * eps)
            scale = max(abs(fd), float(np.abs(dl[t]).max()), 1e-6)
            assert abs(dl[t, e] - fd) <= 2e-2 * scale, (t, e, dl[t, e], fd)


def test_weight_gradient_by_central_differences():
    wl = RAGGED
    inp, ids, w = _case(wl)
    dwgu, dwd = oracle.backward_dw(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w)
    dY = torch.tensor(bf16_to_f64(inp["dy"]))
    rng = np.random.default_rng(1)
    eps = 1e-4

    def loss(wgu64, wd64):
        x = torch.tensor(bf16_to_f64(inp["x"]))
        lg = torch.tensor(inp["logits"].astype(np.float64))
        mask = torch.zeros(lg.shape, dtype=torch.bool)
        mask[torch.arange(wl.T)[:, None], torch.tensor(ids, dtype=torch.long)] = True
        G = torch.softmax(lg.masked_fill(~mask, float("-inf")), 1)
        gu = torch.einsum("th,enh->ten", x, wgu64)
        a = torch.nn.functional.silu(gu[..., :wl.I]) * gu[..., wl.I:]
        return float((torch.einsum("te,tec->tc", G, torch.einsum("ten,ecn->tec", a, wd64)) * dY).sum())

    wgu0 = torch.tensor(bf16_to_f64(inp["wgu"]))
    wd0 = torch.tensor(bf16_to_f64(inp["wd"]))
    for _ in range(8):
        e, n, h = rng.integers(wl.E), rng.integers(2 * wl.I), rng.integers(wl.H)
        a, b = wgu0.clone(), wgu0.clone()
        a[e, n, h] += eps
        b[e, n, h] -= eps
        fd = (loss(a, wd0) - loss(b, wd0)) / (2 * eps)
        got = bf16_to_f64(dwgu)[e, n, h]
        scale = max(abs(fd), float(np.sqrt(np.mean(bf16_to_f64(dwgu)[e] ** 2))))
        assert abs(got - fd) <= 1e-2 * scale, ("dW_gu", e, n, h, got, fd)
        e, c, n = rng.integers(wl.E), rng.integers(wl.H), rng.integers(wl.I)
        a, b = wd0.clone(), wd0.clone()
        a[e, c, n] += eps
        b[e, c, n] -= eps
        fd = (loss(wgu0, a) - loss(wgu0, b)) / (2 * eps)
        got = bf16_to_f64(dwd)[e, c, n]
        scale = max(abs(fd), float(np.sqrt(np.mean(bf16_to_f64(dwd)[e] ** 2))))
        assert abs(got - fd) <= 1e-2 * scale, ("dW_d", e, c, n, got, fd)


def test_single_expert_is_dense_swiglu_mlp():
    wl = synthetic.Workload("single_T40_H128_I64_E1_k1", 40, 128, 64, 1, 1)
    inp, ids, w = _case(wl)
    assert np.all(ids == 0) and np.all(w == 1.0)
    Y = oracle.forward_tokens(inp["x"], inp["wgu"], inp["wd"], ids, w)
    ref = dense_swiglu_mlp_fp64(inp["x"], inp["wgu"][0], inp["wd"][0]).numpy()
    mx, mn = rel_errors(bf16_to_f64(Y), ref)
    assert mx <= ORACLE_MAX_REL and mn <= ORACLE_MEAN_REL
    _, dl = oracle.backward_tokens(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w)
    assert np.all(dl == 0.0)  # k = 1: the single weight is 1 whatever the logit


def test_identical_experts_are_one_dense_mlp():
    wl = synthetic.Workload("same_T64_H128_I64_E6_k3", 64, 128, 64, 6, 3)
    inp, ids, w = _case(wl)
    wgu = np.broadcast_to(inp["wgu"][2], inp["wgu"].shape).copy()
    wd = np.broadcast_to(inp["wd"][2], inp["wd"].shape).copy()
    Y = oracle.forward_tokens(inp["x"], wgu, wd, ids, w)
    ref = dense_swiglu_mlp_fp64(inp["x"], wgu[0], wd[0]).numpy()
    mx, mn = rel_errors(bf16_to_f64(Y), ref)
    assert mx <= ORACLE_MAX_REL and mn <= ORACLE_MEAN_REL
    _, dl = oracle.backward_tokens(inp["x"], inp["dy"], wgu, wd, ids, w)
    # every gamma_j is the same number, so d_logits = w_j*gamma*(1 - sum w) ~ float rounding
    _, dl_ref = oracle.backward_tokens(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w)
    assert np.abs(dl).max() <= 1e-5 * np.abs(dl_ref).max()


def test_identity_expert_roundtrip():
    """f_e(x) = x: dispatch, scale by w, combine returns x within a bf16 ulp or two."""
    wl = TINY
    inp, ids, w = _case(wl)
    d = oracle.dispatch(ids, w, inp["x"], wl.E)
    y = synthetic.f32_to_bf16_bits(synthetic.bf16_bits_to_f32(d["x_perm"]) * d["w_perm"][:, None])
    Y = oracle.combine(y, d["slot_to_row"], wl.T, wl.k)
    x = bf16_to_f64(inp["x"])
    err = np.abs(bf16_to_f64(Y) - x)
    assert np.all(err <= 2.0 ** -7 * np.abs(x) + 1e-30)


def test_empty_expert_weight_gradients_are_exact_zero():
    wl = synthetic.Workload("empty_T32_H64_I64_E10_k2", 32, 64, 64, 10, 2)
    inp, _, _ = _case(wl)
    ids = np.stack([np.arange(32) % 3, 3 + np.arange(32) % 4], 1).astype(np.int32)  # experts 7..9 unused
    w = np.full((32, 2), 0.5, np.float32)
    dwgu, dwd = oracle.backward_dw(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w)
    assert np.all(dwgu[7:] == 0) and np.all(dwd[7:] == 0)
    assert np.any(dwgu[0] != 0) and np.any(dwd[6] != 0)


def test_closed_form_worked_example():
    g = json.load(open(GOLDEN))["layer"]
    b = lambda a: synthetic.f32_to_bf16_bits(np.array(a, np.float32))
    x, wgu, wd, dy = b(g["x"]), b(g["w_gate_up"]), b(g["w_down"]), b(g["dY"])
    ids, w = oracle.route_topk(np.array(g["logits"], np.float32), g["k"])
    np.testing.assert_array_equal(ids, g["ids"])
    np.testing.assert_array_equal(w, np.array(g["w"], np.float32))
    d = oracle.dispatch(ids, w, x, g["E"])
    h, _, _ = oracle.grouped_swiglu_rows(d["x_perm"], d["m_indptr"], wgu, wd, d["w_perm"],
                                         np.arange(2, dtype=np.int32))
    np.testing.assert_array_equal(bf16_to_f64(h).ravel(), g["h"])
    np.testing.assert_array_equal(bf16_to_f64(oracle.forward_tokens(x, wgu, wd, ids, w)), g["Y"])
    dX, dl = oracle.backward_tokens(x, dy, wgu, wd, ids, w)
    np.testing.assert_array_equal(bf16_to_f64(dX), g["dX"])
    np.testing.assert_allclose(dl, g["d_logits"], rtol=1e-6)
    dwgu, dwd = oracle.backward_dw(x, dy, wgu, wd, ids, w)
    np.testing.assert_array_equal(bf16_to_f64(dwgu), g["dW_gate_up"])
    np.testing.assert_array_equal(bf16_to_f64(dwd), g["dW_down"])
