"""GPU parity of the grouped SwiGLU GEMMs, combine and backward against the oracle.

Bar: bit-exact integers; bf16 outputs within max_rel 2e-2 / mean_rel 1e-2 of the
oracle (tests/helpers.py), weight gradients with a per-expert rms floor.
"""
import numpy as np
import pytest
import torch

import mixture_experts_routed_router_gb300 as moe
import oracle
import synthetic
from tests.gpu_util import dw_fp16, to_dev, to_host
from tests.helpers import assert_close, bf16_to_f64, swiglu_factors, off_selection

pytestmark = pytest.mark.gpu

W = synthetic.Workload
CASES = [
    W("tiny_T256_H256_I128_E8_k2", 256, 256, 128, 8, 2),
    W("ragged_T700_H320_I192_E5_k3", 700, 320, 192, 5, 3),          # ragged M, N and gate/up tails
    W("many_T300_H128_I64_E37_k5", 300, 128, 64, 37, 5),             # E not a multiple of 32, tiny groups
    W("zipf_T512_H256_I128_E16_k4", 512, 256, 128, 16, 4, zipf_s=1.2, router_std=0.3),  # skewed + empty experts
    W("single_T200_H128_I128_E1_k1", 200, 128, 128, 1, 1),
    # at least 512 rows per expert: the forward GEMMs run as 2-SM pairs over 256-row tiles
    W("pairs_T2048_H256_I128_E8_k2", 2048, 256, 128, 8, 2),
    W("pairs_zipf_T2048_H320_I192_E4_k2", 2048, 320, 192, 4, 2, zipf_s=1.2, router_std=0.3),  # ragged, skewed
    W("limits_T64_H128_I64_E1024_k32", 64, 128, 64, 1024, 32, router_std=0.3),  # the largest E and k
    # fewer than 192 rows per expert on average, a few experts with 512 or more: the heavy experts run
    # as 2-SM pairs and the rest one CTA per tile (two launches per GEMM); ragged N tails, empty experts
    W("split_zipf_T1024_H320_I192_E64_k8", 1024, 320, 192, 64, 8, zipf_s=1.2, router_std=0.05),
]


MODES = ["x_perm", "gather"]  # expert inputs from the dispatched copy, or gathered by token inside the GEMMs


def _run_forward(wl, inp, save_gu=True, mode="x_perm"):
    ids, w = moe.route_topk(to_dev(inp["logits"]), wl.k)
    x = to_dev(inp["x"])
    wgu, wd = to_dev(inp["wgu"]), to_dev(inp["wd"])
    if mode == "gather":
        d = moe.dispatch(ids, w, None, wl.E)
        h, gu, y_perm = moe.grouped_swiglu_fwd_gather(x, d["row_to_slot"], wl.k, d["m_indptr"], wgu, wd, d["w_perm"],
                                                      save_gu=save_gu)
    else:
        d = moe.dispatch(ids, w, x, wl.E)
        h, gu, y_perm = moe.grouped_swiglu_fwd(d["x_perm"], d["m_indptr"], wgu, wd, d["w_perm"], save_gu=save_gu)
    Y = moe.combine(y_perm, d["slot_to_row"], wl.T, wl.k)
    return dict(ids=ids, w=w, x=x, d=d, wgu=wgu, wd=wd, h=h, gu=gu, y_perm=y_perm, Y=Y, mode=mode)


def _run_backward(g, dy, **kw):
    d = g["d"]
    if g["mode"] == "gather":
        return moe.bwd_dx_dw_gather(dy, g["x"], g["h"], g["gu"], g["ids"], g["w"], d["m_indptr"], d["row_to_slot"],
                                    d["slot_to_row"], d["w_perm"], g["wgu"], g["wd"], **kw)
    return moe.bwd_dx_dw(dy, d["x_perm"], g["h"], g["gu"], g["ids"], g["w"], d["m_indptr"], d["row_to_slot"],
                         d["slot_to_row"], d["w_perm"], g["wgu"], g["wd"], **kw)


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("mode", MODES)
def test_forward_parity(wl, mode):
    inp = synthetic.make_inputs(wl)
    g = _run_forward(wl, inp, mode=mode)
    assert moe.device_error() == 0
    ids, w = oracle.route_topk(inp["logits"], wl.k)
    np.testing.assert_array_equal(to_host(g["ids"]), ids)
    ref = oracle.dispatch(ids, w, inp["x"], wl.E)
    np.testing.assert_array_equal(to_host(g["d"]["m_indptr"]), ref["m_indptr"])
    rows = np.arange(wl.R, dtype=np.int32)
    # the oracle's expert MLP on the GPU's own dispatched inputs (identical to its own by the check above)
    h, gu, y = oracle.grouped_swiglu_rows(ref["x_perm"], ref["m_indptr"], inp["wgu"], inp["wd"],
                                          to_host(g["d"]["w_perm"]), rows)
    assert_close(bf16_to_f64(to_host(g["h"])), bf16_to_f64(h), "h_perm")
    # saved SwiGLU derivative factors from the fp32 accumulators: summation order only
    assert_close(to_host(g["gu"]), swiglu_factors(gu), "gu_perm", max_rel=1e-3, mean_rel=1e-4)
    assert_close(bf16_to_f64(to_host(g["y_perm"])), bf16_to_f64(y), "y_perm")
    Y = oracle.forward_tokens(inp["x"], inp["wgu"], inp["wd"], ids, w)
    assert_close(bf16_to_f64(to_host(g["Y"])), bf16_to_f64(Y), "Y")


def test_combine_is_bit_exact():
    wl = CASES[1]
    inp = synthetic.make_inputs(wl, want=("x", "logits"))
    ids, w = oracle.route_topk(inp["logits"], wl.k)
    ref = oracle.dispatch(ids, w, inp["x"], wl.E)
    y_perm = synthetic.normal_bf16((wl.R, wl.H), seed=3, stream=21, sigma=1.0)
    Y = moe.combine(to_dev(y_perm), to_dev(ref["slot_to_row"]), wl.T, wl.k)
    np.testing.assert_array_equal(to_host(Y), oracle.combine(y_perm, ref["slot_to_row"], wl.T, wl.k))


def test_identity_expert_roundtrip_on_gpu():
    """Dispatch, scale each row by its weight (the down epilogue's job), combine: returns x."""
    wl = CASES[0]
    inp = synthetic.make_inputs(wl, want=("x", "logits"))
    ids, w = moe.route_topk(to_dev(inp["logits"]), wl.k)
    d = moe.dispatch(ids, w, to_dev(inp["x"]), wl.E)
    y_perm = (d["x_perm"].float() * d["w_perm"][:, None]).to(torch.bfloat16)
    Y = moe.combine(y_perm, d["slot_to_row"], wl.T, wl.k)
    x = bf16_to_f64(inp["x"])
    assert np.all(np.abs(bf16_to_f64(to_host(Y)) - x) <= 2.0 ** -7 * np.abs(x) + 1e-30)


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("save_gu", [True, False], ids=["saved_gu", "recomputed_gu"])
@pytest.mark.parametrize("mode", MODES)
def test_backward_parity(wl, save_gu, mode):
    inp = synthetic.make_inputs(wl)
    g = _run_forward(wl, inp, save_gu=save_gu, mode=mode)
    dx, dwgu, dwd, dl = _run_backward(g, to_dev(inp["dy"]))
    assert moe.device_error() == 0
    ids, w = oracle.route_topk(inp["logits"], wl.k)
    rdx, rdl = oracle.backward_tokens(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w)
    rdwgu, rdwd = oracle.backward_dw(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w)
    assert_close(bf16_to_f64(to_host(dx)), bf16_to_f64(rdx), "dX")
    dl_h = to_host(dl)
    assert_close(dl_h, rdl, "d_logits")
    assert np.all(dl_h[off_selection(ids, wl.E)] == 0)  # exact zeros off the selection
    assert_close(bf16_to_f64(to_host(dwgu)), bf16_to_f64(rdwgu), "dW_gate_up", per_expert=True)
    assert_close(bf16_to_f64(to_host(dwd)), bf16_to_f64(rdwd), "dW_down", per_expert=True)
    empty = np.nonzero(np.bincount(ids.ravel(), minlength=wl.E) == 0)[0]
    assert np.all(to_host(dwgu)[empty] == 0) and np.all(to_host(dwd)[empty] == 0)


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_gathered_inputs_match_the_dispatched_copy_bitwise(wl):
    """Gathering rows by token inside the GEMMs feeds the tensor cores the same bytes as x_perm.
    (The gathered backward always takes the hi / lo weight-gradient operands, so the x_perm one is
    compared with its fp16 pass off.)"""
    inp = synthetic.make_inputs(wl)
    a = _run_forward(wl, inp, mode="x_perm")
    b = _run_forward(wl, inp, mode="gather")
    for key in ("h", "gu", "y_perm", "Y"):
        assert torch.equal(a[key], b[key]), key
    dy = to_dev(inp["dy"])
    with dw_fp16(False):
        ra = _run_backward(a, dy)
    for u, v, name in zip(ra, _run_backward(b, dy), ("dX", "dW_gate_up", "dW_down", "d_logits")):
        assert torch.equal(u, v), name
    assert moe.device_error() == 0


def test_backward_is_deterministic():
    wl = CASES[3]
    inp = synthetic.make_inputs(wl)
    g = _run_forward(wl, inp)
    d = g["d"]
    args = (to_dev(inp["dy"]), d["x_perm"], g["h"], g["gu"], g["ids"], g["w"], d["m_indptr"], d["row_to_slot"],
            d["slot_to_row"], d["w_perm"], g["wgu"], g["wd"])
    a = moe.bwd_dx_dw(*args)
    b = moe.bwd_dx_dw(*args)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


@pytest.mark.parametrize("mode", MODES)
def test_zero_tokens_gives_zero_weight_gradients(mode):
    wl = W("zero_T0_H128_I64_E4_k2", 0, 128, 64, 4, 2)
    E, H, I = wl.E, wl.H, wl.I
    z = lambda *s, dt=torch.bfloat16: torch.empty(s, dtype=dt, device="cuda")
    x = z(0, H)
    d = moe.dispatch(z(0, 2, dt=torch.int32), z(0, 2, dt=torch.float32), x, E)
    wgu = torch.randn(E, 2 * I, H, device="cuda").to(torch.bfloat16)
    wd = torch.randn(E, H, I, device="cuda").to(torch.bfloat16)
    if mode == "gather":
        h, gu, y = moe.grouped_swiglu_fwd_gather(x, d["row_to_slot"], 2, d["m_indptr"], wgu, wd, d["w_perm"])
    else:
        h, gu, y = moe.grouped_swiglu_fwd(d["x_perm"], d["m_indptr"], wgu, wd, d["w_perm"])
    out = dict(dw_gate_up=torch.full((E, 2 * I, H), 7.0, device="cuda").to(torch.bfloat16),
               dw_down=torch.full((E, H, I), 7.0, device="cuda").to(torch.bfloat16))
    bwd = moe.bwd_dx_dw_gather if mode == "gather" else moe.bwd_dx_dw
    dx, dwgu, dwd, dl = bwd(z(0, H), x if mode == "gather" else d["x_perm"], h, gu, z(0, 2, dt=torch.int32),
                            z(0, 2, dt=torch.float32), d["m_indptr"], d["row_to_slot"], d["slot_to_row"],
                            d["w_perm"], wgu, wd, out=out)
    assert moe.device_error() == 0
    assert torch.count_nonzero(dwgu) == 0 and torch.count_nonzero(dwd) == 0


def test_bad_row_to_slot_is_flagged_not_faulted():
    wl = CASES[0]
    inp = synthetic.make_inputs(wl)
    g = _run_forward(wl, inp, mode="gather")
    assert moe.device_error() == 0
    bad = g["d"]["row_to_slot"].clone()
    bad[5] = wl.R + 7
    bad[9] = -3
    moe.grouped_swiglu_fwd_gather(g["x"], bad, wl.k, g["d"]["m_indptr"], g["wgu"], g["wd"], g["d"]["w_perm"])
    assert moe.device_error() & 0x2


def test_bad_indptr_is_flagged_not_faulted():
    wl = CASES[0]
    inp = synthetic.make_inputs(wl)
    g = _run_forward(wl, inp)
    bad = g["d"]["m_indptr"].clone()
    bad[3] = bad[4] + 5  # not monotone
    moe.grouped_swiglu_fwd(g["d"]["x_perm"], bad, g["wgu"], g["wd"], g["d"]["w_perm"])
    assert moe.device_error() & 0x4
