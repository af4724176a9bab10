"""GPU parity of the activation variants (bounded SwiGLU, SwiGLU-OAI, GeGLU, ReGLU, and the two-weight
ReLU² experts) against the oracle.

LightMoE README, "Compatibility" / "Highlights" name the variants.  The CUDA path runs them through
liger_moe_grouped_glu_fwd (the gate/up epilogue computes h and the fp32 derivative factors
dh/dg, dh/du) and liger_moe_bwd_dx_dw_glu (which recomputes the factors with the same activation
when they were not saved).  Same bar as the SwiGLU path: bf16 outputs within max_rel 2e-2 /
mean_rel 1e-2 of the oracle, weight gradients per expert.

A clamp or a ReLU makes a factor jump where g or u crosses the clamp (or 0); the GPU's fp32 sums and
the oracle's run in different orders, so the two may fall on opposite sides for an element within
rounding of the edge.  The factor comparison leaves out elements whose pre-activation lies within
1e-3 (relative) of an edge; every other element is compared.
"""
import numpy as np
import pytest
import torch

import mixture_experts_routed_router_gb300 as moe
import oracle
import synthetic
from tests.gpu_util import to_dev, to_host
from tests.helpers import assert_close, bf16_to_f64, gated_act_torch, off_selection

pytestmark = pytest.mark.gpu

W = synthetic.Workload
CASES = [
    W("tiny_T256_H256_I128_E8_k2", 256, 256, 128, 8, 2),
    W("ragged_T700_H320_I192_E5_k3", 700, 320, 192, 5, 3),
    W("zipf_T512_H256_I128_E16_k4", 512, 256, 128, 16, 4, zipf_s=1.2, router_std=0.3),
    W("pairs_T2048_H256_I128_E8_k2", 2048, 256, 128, 8, 2),  # 512 rows per expert: 2-SM pair GEMMs
]
# small clamps so that the synthetic pre-activations cross them
VARIANTS = [("swiglu_bounded", 0.75), ("swiglu_oai", 1.0), ("geglu", 0.0), ("reglu", 0.0)]


def gated_factors_fp64(gu: np.ndarray, act: str, clamp: float) -> np.ndarray:
    """[dh/dg | dh/du] of the activation at the oracle's accumulators [g | u] (fp64 autograd)."""
    t = torch.tensor(np.asarray(gu, dtype=np.float64), requires_grad=True)
    I = t.shape[1] // 2
    gated_act_torch(t[:, :I], t[:, I:], act, clamp).sum().backward()
    return t.grad.numpy()


def edge_mask(gu: np.ndarray, act: str, clamp: float) -> np.ndarray:
    """True where g or u lies within rounding of a point where the factors jump ([R, 2I], both halves)."""
    I = gu.shape[1] // 2
    g, u = gu[:, :I].astype(np.float64), gu[:, I:].astype(np.float64)
    near = np.zeros_like(g, dtype=bool)
    if act in ("swiglu_bounded", "swiglu_oai"):
        near |= np.abs(g - clamp) <= 1e-3 * clamp
        near |= np.abs(np.abs(u) - clamp) <= 1e-3 * clamp
    if act == "reglu":
        near |= np.abs(g) <= 1e-3 * (np.abs(g).max() + 1e-30)
    return np.concatenate([near, near], axis=1)


def _forward(wl, inp, act, clamp, save_gu=True):
    ids, w = moe.route_topk(to_dev(inp["logits"]), wl.k)
    x = to_dev(inp["x"])
    wgu, wd = to_dev(inp["wgu"]), to_dev(inp["wd"])
    d = moe.dispatch(ids, w, x, wl.E)
    h, gu, y_perm = moe.grouped_glu_fwd(d["x_perm"], d["m_indptr"], wgu, wd, d["w_perm"], act, clamp,
                                        save_gu=save_gu)
    Y = moe.combine(y_perm, d["slot_to_row"], wl.T, wl.k)
    return dict(ids=ids, w=w, d=d, wgu=wgu, wd=wd, h=h, gu=gu, y_perm=y_perm, Y=Y)


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("act,clamp", VARIANTS)
def test_forward_parity(wl, act, clamp):
    inp = synthetic.make_inputs(wl)
    g = _forward(wl, inp, act, clamp)
    assert moe.device_error() == 0
    ids, w = oracle.route_topk(inp["logits"], wl.k)
    ref = oracle.dispatch(ids, w, inp["x"], wl.E)
    np.testing.assert_array_equal(to_host(g["d"]["m_indptr"]), ref["m_indptr"])
    rows = np.arange(wl.R, dtype=np.int32)
    h, gu, y = oracle.grouped_swiglu_rows(ref["x_perm"], ref["m_indptr"], inp["wgu"], inp["wd"],
                                          to_host(g["d"]["w_perm"]), rows, act=act, clamp=clamp)
    assert_close(bf16_to_f64(to_host(g["h"])), bf16_to_f64(h), f"h_perm[{act}]")
    keep = ~edge_mask(gu, act, clamp)
    assert keep.mean() > 0.99
    got_f, ref_f = to_host(g["gu"]).astype(np.float64), gated_factors_fp64(gu, act, clamp)
    assert_close(got_f[keep], ref_f[keep], f"gu_perm[{act}]", max_rel=1e-3, mean_rel=1e-4)
    if act in ("swiglu_bounded", "swiglu_oai", "reglu"):  # the blocked gradients are exact zeros
        assert np.all(got_f[keep & (ref_f == 0)] == 0)
        assert (ref_f[keep] == 0).mean() > 0.01  # the clamp / ReLU branches were exercised
    assert_close(bf16_to_f64(to_host(g["y_perm"])), bf16_to_f64(y), f"y_perm[{act}]")
    Y = oracle.forward_tokens(inp["x"], inp["wgu"], inp["wd"], ids, w, act=act, clamp=clamp)
    assert_close(bf16_to_f64(to_host(g["Y"])), bf16_to_f64(Y), f"Y[{act}]")


@pytest.mark.parametrize("wl", CASES[1:], ids=lambda w: w.name)
@pytest.mark.parametrize("save_gu", [True, False], ids=["saved_gu", "recomputed_gu"])
@pytest.mark.parametrize("act,clamp", VARIANTS)
def test_backward_parity(wl, save_gu, act, clamp):
    inp = synthetic.make_inputs(wl)
    g = _forward(wl, inp, act, clamp, save_gu=save_gu)
    d = g["d"]
    dx, dwgu, dwd, dl = moe.bwd_dx_dw_glu(to_dev(inp["dy"]), d["x_perm"], g["h"], g["gu"], g["ids"], g["w"],
                                          d["m_indptr"], d["row_to_slot"], d["slot_to_row"], d["w_perm"], g["wgu"],
                                          g["wd"], act, clamp)
    assert moe.device_error() == 0
    ids, w = oracle.route_topk(inp["logits"], wl.k)
    kw = dict(act=act, clamp=clamp)
    rdx, rdl = oracle.backward_tokens(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w, **kw)
    rdwgu, rdwd = oracle.backward_dw(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w, **kw)
    assert_close(bf16_to_f64(to_host(dx)), bf16_to_f64(rdx), f"dX[{act}]")
    dl_h = to_host(dl)
    assert_close(dl_h, rdl, f"d_logits[{act}]")
    assert np.all(dl_h[off_selection(ids, wl.E)] == 0)
    assert_close(bf16_to_f64(to_host(dwgu)), bf16_to_f64(rdwgu), f"dW_gate_up[{act}]", per_expert=True)
    assert_close(bf16_to_f64(to_host(dwd)), bf16_to_f64(rdwd), f"dW_down[{act}]", per_expert=True)


def test_wide_clamp_reduces_to_swiglu():
    """A clamp above every pre-activation leaves bounded SwiGLU equal to SwiGLU: same h, factors, y."""
    wl = CASES[1]
    inp = synthetic.make_inputs(wl)
    a = _forward(wl, inp, "swiglu_bounded", 1e30)
    d = a["d"]
    h, gu, y = moe.grouped_swiglu_fwd(d["x_perm"], d["m_indptr"], a["wgu"], a["wd"], d["w_perm"])
    assert moe.device_error() == 0
    np.testing.assert_allclose(bf16_to_f64(to_host(a["h"])), bf16_to_f64(to_host(h)), rtol=2.0 ** -7, atol=0)
    np.testing.assert_allclose(to_host(a["gu"]), to_host(gu), rtol=1e-6, atol=1e-30)
    np.testing.assert_allclose(bf16_to_f64(to_host(a["y_perm"])), bf16_to_f64(to_host(y)), rtol=2.0 ** -7,
                               atol=1e-30)


def test_glu_entry_with_swiglu_is_the_swiglu_path_bitwise():
    wl = CASES[0]
    inp = synthetic.make_inputs(wl)
    a = _forward(wl, inp, "swiglu", 0.0)
    d = a["d"]
    h, gu, y = moe.grouped_swiglu_fwd(d["x_perm"], d["m_indptr"], a["wgu"], a["wd"], d["w_perm"])
    assert torch.equal(a["h"], h) and torch.equal(a["gu"], gu) and torch.equal(a["y_perm"], y)


# ------------------------------------------------------------------ ReLU² (two-weight experts)
# LightMoE README, "MoE inference": ReLU² experts hold an up and a down weight, no gate.  The up
# weight W_up [E, I, H] takes the place of W_gate_up; here it is the gate half of the synthetic
# W_gu (same N(0, 1/sqrt(H)) init).  gu_perm [R, I] holds dh/da = 2 max(a, 0).


def _relu2_inputs(wl):
    inp = synthetic.make_inputs(wl)
    inp["wgu"] = np.ascontiguousarray(inp["wgu"][:, : wl.I])
    return inp


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_relu2_forward_parity(wl):
    inp = _relu2_inputs(wl)
    g = _forward(wl, inp, "relu2", 0.0)
    assert moe.device_error() == 0
    assert tuple(g["gu"].shape) == (wl.R, wl.I)
    ids, w = oracle.route_topk(inp["logits"], wl.k)
    ref = oracle.dispatch(ids, w, inp["x"], wl.E)
    rows = np.arange(wl.R, dtype=np.int32)
    h, a, y = oracle.grouped_swiglu_rows(ref["x_perm"], ref["m_indptr"], inp["wgu"], inp["wd"],
                                         to_host(g["d"]["w_perm"]), rows, act="relu2")
    assert_close(bf16_to_f64(to_host(g["h"])), bf16_to_f64(h), "h_perm[relu2]")
    # dh/da = 2 max(a, 0) at the oracle's fp32 a; elements within rounding of a = 0 may take either side
    a64 = a.astype(np.float64)
    keep = np.abs(a64) > 1e-3 * np.abs(a64).max()
    assert keep.mean() > 0.99
    got_f, ref_f = to_host(g["gu"]).astype(np.float64), 2.0 * np.maximum(a64, 0.0)
    assert_close(got_f[keep], ref_f[keep], "gu_perm[relu2]", max_rel=1e-3, mean_rel=1e-4)
    assert np.all(got_f[keep & (a64 < 0)] == 0)
    assert 0.3 < (a64 < 0).mean() < 0.7  # both branches of the ReLU are exercised
    assert_close(bf16_to_f64(to_host(g["y_perm"])), bf16_to_f64(y), "y_perm[relu2]")
    Y = oracle.forward_tokens(inp["x"], inp["wgu"], inp["wd"], ids, w, act="relu2")
    assert_close(bf16_to_f64(to_host(g["Y"])), bf16_to_f64(Y), "Y[relu2]")


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("save_gu", [True, False], ids=["saved_gu", "recomputed_gu"])
def test_relu2_backward_parity(wl, save_gu):
    inp = _relu2_inputs(wl)
    g = _forward(wl, inp, "relu2", 0.0, save_gu=save_gu)
    d = g["d"]
    dx, dwup, dwd, dl = moe.bwd_dx_dw_glu(to_dev(inp["dy"]), d["x_perm"], g["h"], g["gu"], g["ids"], g["w"],
                                          d["m_indptr"], d["row_to_slot"], d["slot_to_row"], d["w_perm"], g["wgu"],
                                          g["wd"], "relu2")
    assert moe.device_error() == 0
    assert tuple(dwup.shape) == (wl.E, wl.I, wl.H)
    ids, w = oracle.route_topk(inp["logits"], wl.k)
    rdx, rdl = oracle.backward_tokens(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w, act="relu2")
    rdwup, rdwd = oracle.backward_dw(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w, act="relu2")
    assert_close(bf16_to_f64(to_host(dx)), bf16_to_f64(rdx), "dX[relu2]")
    dl_h = to_host(dl)
    assert_close(dl_h, rdl, "d_logits[relu2]")
    assert np.all(dl_h[off_selection(ids, wl.E)] == 0)
    assert_close(bf16_to_f64(to_host(dwup)), bf16_to_f64(rdwup), "dW_up[relu2]", per_expert=True)
    assert_close(bf16_to_f64(to_host(dwd)), bf16_to_f64(rdwd), "dW_down[relu2]", per_expert=True)


def test_relu2_rejects_a_gated_weight_shape():
    """The binding checks W_up's shape against I from W_down: a [E, 2I, H] weight is refused for relu2."""
    wl = CASES[0]
    inp = synthetic.make_inputs(wl)
    ids, w = moe.route_topk(to_dev(inp["logits"]), wl.k)
    d = moe.dispatch(ids, w, to_dev(inp["x"]), wl.E)
    with pytest.raises(ValueError):
        moe.grouped_glu_fwd(d["x_perm"], d["m_indptr"], to_dev(inp["wgu"]), to_dev(inp["wd"]), d["w_perm"], "relu2")
