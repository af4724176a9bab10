"""Pins for the oracle's activation variants (bounded SwiGLU, SwiGLU-OAI, GeGLU, ReGLU, ReLU²), CPU only.

LightMoE README, "Compatibility" and "Highlights" name the activations; their formulas are the
plainest published forms (written out in tests/helpers.py gated_act_torch, independently of the
oracle's C++).  Expected values come from that fp64 torch form (dense over all experts, autograd for
the gradients) and from closed-form values at chosen points; the clamp values here are small so that
the clamp branches are exercised by the synthetic N(0, 1) pre-activations.  ReLU² experts hold two
weights (LightMoE README, "MoE inference"); its up weight [E, I, H] is the gate half of the
synthetic W_gu.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic
from tests.helpers import bf16_to_f64, dense_layer_fp64, rel_errors, rel_errors_per_expert

ORACLE_MAX_REL = 1.5e-2
ORACLE_MEAN_REL = 3e-3

VARIANTS = [("swiglu_bounded", 0.75), ("swiglu_oai", 1.0), ("geglu", 0.0), ("reglu", 0.0), ("relu2", 0.0)]
RAGGED = synthetic.Workload("ragged_T50_H64_I64_E5_k3", 50, 64, 64, 5, 3)


def _case(wl, act="swiglu"):
    inp = synthetic.make_inputs(wl)
    if act == "relu2":  # the two-weight form: the up weight is the gate half of W_gu
        inp["wgu"] = np.ascontiguousarray(inp["wgu"][:, : wl.I])
    ids, w = oracle.route_topk(inp["logits"], wl.k)
    return inp, ids, w


@pytest.mark.parametrize("act,clamp", VARIANTS)
def test_forward_matches_fp64_dense(act, clamp):
    inp, ids, w = _case(RAGGED, act)
    Y = oracle.forward_tokens(inp["x"], inp["wgu"], inp["wd"], ids, w, act=act, clamp=clamp)
    Yd, _ = dense_layer_fp64(inp["x"], inp["wgu"], inp["wd"], inp["logits"], ids, act=act, clamp=clamp)
    mx, mn = rel_errors(bf16_to_f64(Y), Yd.numpy())
    assert mx <= ORACLE_MAX_REL and mn <= ORACLE_MEAN_REL, (mx, mn)


@pytest.mark.parametrize("act,clamp", VARIANTS)
def test_backward_matches_fp64_autograd(act, clamp):
    inp, ids, w = _case(RAGGED, act)
    dX, dl = oracle.backward_tokens(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w, act=act, clamp=clamp)
    dwgu, dwd = oracle.backward_dw(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w, act=act, clamp=clamp)
    Yd, leaves = dense_layer_fp64(inp["x"], inp["wgu"], inp["wd"], inp["logits"], ids, requires_grad=True,
                                  act=act, clamp=clamp)
    (Yd * torch.tensor(bf16_to_f64(inp["dy"]))).sum().backward()
    for name, got, ref, metric in (("dX", bf16_to_f64(dX), leaves["x"].grad, rel_errors),
                                   ("dW_gu", bf16_to_f64(dwgu), leaves["wgu"].grad, rel_errors_per_expert),
                                   ("dW_d", bf16_to_f64(dwd), leaves["wd"].grad, rel_errors_per_expert),
                                   ("d_logits", dl, leaves["logits"].grad, rel_errors)):
        mx, mn = metric(got, ref.numpy())
        assert mx <= ORACLE_MAX_REL and mn <= ORACLE_MEAN_REL, (name, mx, mn)


@pytest.mark.parametrize("act,clamp", VARIANTS)
def test_grouped_rows_agree_with_per_token_forward(act, clamp):
    inp, ids, w = _case(RAGGED, act)
    d = oracle.dispatch(ids, w, inp["x"], RAGGED.E)
    rows = np.arange(RAGGED.R, dtype=np.int32)
    _, _, y = oracle.grouped_swiglu_rows(d["x_perm"], d["m_indptr"], inp["wgu"], inp["wd"], d["w_perm"], rows,
                                         act=act, clamp=clamp)
    Yc = oracle.combine(y, d["slot_to_row"], RAGGED.T, RAGGED.k)
    Yt = oracle.forward_tokens(inp["x"], inp["wgu"], inp["wd"], ids, w, act=act, clamp=clamp)
    np.testing.assert_array_equal(Yc, Yt)


def _one_hot_layer(g_vals, u_vals, gated=True):
    """One token, one expert, k = 1: x = e_0, W_gu[:, 0] = (g, u), W_d = identity.  Then
    g, u are exactly the given (bf16) values and Y[n] = bf16(act(g[n], u[n])).  Not gated:
    W_up[:, 0] = g and Y[n] = bf16(act(g[n]))."""
    I = len(g_vals)
    H = I
    x = np.zeros((1, H), np.float32)
    x[0, 0] = 1.0
    wgu = np.zeros((1, 2 * I if gated else I, H), np.float32)
    wgu[0, :I, 0] = g_vals
    if gated:
        wgu[0, I:, 0] = u_vals
    wd = np.eye(H, I, dtype=np.float32)[None]
    bits = synthetic.f32_to_bf16_bits
    return bits(x), bits(wgu), bits(wd), np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32)


def _gelu_tanh(g):
    return 0.5 * g * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (g + 0.044715 * g ** 3)))


def _sig(a):
    return 1.0 / (1.0 + math.exp(-a))


CLOSED_FORM = [
    # (act, clamp, g, u, exact h)
    ("swiglu_bounded", 10.0, 12.0, 3.0, 10.0 * _sig(10.0) * 3.0),      # gate clamped from above
    ("swiglu_bounded", 10.0, 2.0, -16.0, 2.0 * _sig(2.0) * -10.0),     # up clamped from below
    ("swiglu_bounded", 10.0, -20.0, 2.0, -20.0 * _sig(-20.0) * 2.0),   # gate not clamped from below
    ("swiglu_bounded", 10.0, 1.5, 0.5, 1.5 * _sig(1.5) * 0.5),         # inside: plain SwiGLU
    ("swiglu_oai", 7.0, 8.0, 0.5, 7.0 * _sig(1.702 * 7.0) * 1.5),      # limit on the gate
    ("swiglu_oai", 7.0, 1.0, 0.0, 1.0 * _sig(1.702) * 1.0),            # the +1 on the linear part
    ("swiglu_oai", 7.0, -2.0, 9.0, -2.0 * _sig(-3.404) * 8.0),         # linear part clamped at the limit
    ("geglu", 0.0, 1.0, 1.0, _gelu_tanh(1.0)),
    ("geglu", 0.0, -2.0, 3.0, _gelu_tanh(-2.0) * 3.0),
    ("reglu", 0.0, -2.0, 5.0, 0.0),
    ("reglu", 0.0, 3.0, 2.0, 6.0),
    ("relu2", 0.0, 3.0, 0.0, 9.0),
    ("relu2", 0.0, -2.0, 0.0, 0.0),
    ("relu2", 0.0, 0.75, 0.0, 0.5625),
]


@pytest.mark.parametrize("act,clamp,g,u,h", CLOSED_FORM)
def test_closed_form_values(act, clamp, g, u, h):
    x, wgu, wd, ids, w = _one_hot_layer([g], [u], gated=act != "relu2")
    Y = oracle.forward_tokens(x, wgu, wd, ids, w, act=act, clamp=clamp)
    got = float(bf16_to_f64(Y)[0, 0])
    # float evaluation then one bf16 rounding: within one bf16 ulp of the exact value
    assert abs(got - h) <= 2.0 ** -8 * max(abs(h), 1e-30) + 1e-30, (got, h)


def test_bounded_swiglu_with_a_wide_clamp_is_swiglu():
    inp, ids, w = _case(RAGGED)
    a = oracle.forward_tokens(inp["x"], inp["wgu"], inp["wd"], ids, w, act="swiglu_bounded", clamp=1e6)
    b = oracle.forward_tokens(inp["x"], inp["wgu"], inp["wd"], ids, w)
    np.testing.assert_array_equal(a, b)


def test_unknown_activation_is_rejected():
    inp, ids, w = _case(RAGGED)
    with pytest.raises(ValueError):
        oracle.forward_tokens(inp["x"], inp["wgu"], inp["wd"], ids, w, act="relu3")


def test_relu2_gradient_closed_form():
    """One token, one expert, k = 1, W_d = identity, dY = e_0: dX[0] = 2 relu(g) W_up[0, 0] and
    dW_up[0, 0] = 2 relu(g) x[0] = 2 relu(g) (x = e_0), both exact in bf16 for these values."""
    for g, dxv in ((3.0, 6.0 * 3.0), (-2.0, 0.0), (0.5, 1.0 * 0.5)):
        x, wup, wd, ids, w = _one_hot_layer([g], [0.0], gated=False)
        dy = synthetic.f32_to_bf16_bits(np.array([[1.0]], np.float32))
        dX, dl = oracle.backward_tokens(x, dy, wup, wd, ids, w, act="relu2")
        dwup, dwd = oracle.backward_dw(x, dy, wup, wd, ids, w, act="relu2")
        assert float(bf16_to_f64(dX)[0, 0]) == dxv
        assert dwup.shape == (1, 1, 1) and float(bf16_to_f64(dwup)[0, 0, 0]) == 2.0 * max(g, 0.0)
        assert float(bf16_to_f64(dwd)[0, 0, 0]) == max(g, 0.0) ** 2
        assert dl[0, 0] == 0.0  # k = 1
