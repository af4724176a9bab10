"""The single fp16 pass of the heavy experts' weight gradients (liger_moe_set_dw_fp16).

Experts with at least 384 rows (batches of R >= 32768 routed rows, gated experts, expert-major
inputs) take dW_gate_up and dW_down in one fp16 MMA per K step: the x and dY rows scaled by powers
of two from their largest magnitudes (exact), dgu and w h rounded to fp16 (11 significant bits)
instead of split into bf16 hi + lo parts.  Checked here, on a skewed batch with both kinds of
expert:
- both precisions match the oracle within the bar;
- the fp16 pass is taken exactly by the heavy experts: their gradients differ from the hi / lo
  run, while dX, d_logits and the light experts' gradients are bit-identical;
- an expert whose scaled dgu leaves the fp16 window (here: its W_down scaled by 2^40, so its dgu
  overflows, or by 2^-40, so its dgu would be subnormal) falls back to the hi / lo parts: it matches
  the oracle and the hi / lo run in all but a few elements (the same products in fp32, the hi and
  lo parts summed as two passes over its rows instead of interleaved, so a rounding of the bf16
  result rarely flips), while the other heavy experts keep the fp16 pass (11-bit dgu: about one
  element in ten rounds differently);
- the pass is deterministic.
"""
import numpy as np
import pytest
import torch

import mixture_experts_routed_router_gb300 as moe
import oracle
import synthetic
from tests.gpu_util import dw_fp16, to_dev, to_host
from tests.helpers import assert_close, bf16_to_f64

pytestmark = pytest.mark.gpu

WL = synthetic.Workload("f16_zipf_T4096_H320_I192_E64_k8", 4096, 320, 192, 64, 8, zipf_s=1.2, router_std=0.05)
HEAVY_ROWS = 384


def _layer(inp, wd=None):
    wl = WL
    ids, w = moe.route_topk(to_dev(inp["logits"]), wl.k)
    x, wgu = to_dev(inp["x"]), to_dev(inp["wgu"])
    wd = to_dev(inp["wd"]) if wd is None else wd
    d = moe.dispatch(ids, w, x, wl.E)
    h, gu, _ = moe.grouped_swiglu_fwd(d["x_perm"], d["m_indptr"], wgu, wd, d["w_perm"])
    args = (to_dev(inp["dy"]), d["x_perm"], h, gu, ids, w, d["m_indptr"], d["row_to_slot"], d["slot_to_row"],
            d["w_perm"], wgu, wd)
    counts = to_host(d["counts"])
    return args, counts


def _oracle_check(inp, out, wd_host=None):
    wd = inp["wd"] if wd_host is None else wd_host
    ids, w = oracle.route_topk(inp["logits"], WL.k)
    rdwgu, rdwd = oracle.backward_dw(inp["x"], inp["dy"], inp["wgu"], wd, ids, w)
    _, dwgu, dwd, _ = out
    assert_close(bf16_to_f64(to_host(dwgu)), bf16_to_f64(rdwgu), "dW_gate_up", per_expert=True)
    assert_close(bf16_to_f64(to_host(dwd)), bf16_to_f64(rdwd), "dW_down", per_expert=True)


def _differs(a, b, experts):
    return [bool((a[e] != b[e]).any()) for e in experts]


def _flipped(a, b):
    """Fraction of elements whose bf16 bits differ."""
    return float(np.mean(a != b))


def test_heavy_experts_take_the_fp16_pass_and_match_the_oracle():
    inp = synthetic.make_inputs(WL)
    args, counts = _layer(inp)
    heavy = np.nonzero(counts >= HEAVY_ROWS)[0]
    light = np.nonzero((counts > 0) & (counts < HEAVY_ROWS))[0]
    assert len(heavy) >= 2 and len(light) >= 2, counts
    f16 = moe.bwd_dx_dw(*args)
    with dw_fp16(False):
        hilo = moe.bwd_dx_dw(*args)
    assert moe.device_error() == 0
    _oracle_check(inp, f16)
    _oracle_check(inp, hilo)
    for name, i in (("dX", 0), ("d_logits", 3)):
        assert torch.equal(f16[i], hilo[i]), name
    for i, name in ((1, "dW_gate_up"), (2, "dW_down")):
        a, b = to_host(f16[i]), to_host(hilo[i])
        assert not any(_differs(a, b, light)), f"{name}: a light expert left the hi / lo path"
        assert all(_differs(a, b, heavy)), f"{name}: a heavy expert did not take the fp16 pass"
    again = moe.bwd_dx_dw(*args)
    for u, v in zip(f16, again):
        assert torch.equal(u, v)


@pytest.mark.parametrize("scale", [2.0 ** 40, 2.0 ** -40], ids=["overflow", "too_small"])
def test_an_expert_outside_the_fp16_window_falls_back_to_hi_lo(scale):
    inp = synthetic.make_inputs(WL)
    _, counts = _layer(inp)
    heavy = np.nonzero(counts >= HEAVY_ROWS)[0]
    assert len(heavy) >= 2, counts
    big = int(np.argmax(counts))
    wd = to_dev(inp["wd"])
    # exact in bf16: the expert's dgu scales with its W_down, and its largest scaled fp16 magnitude
    # leaves the window (overflow above 65504, or below 2^-6 where values would lose precision)
    wd[big] *= scale
    args, _ = _layer(inp, wd=wd)
    f16 = moe.bwd_dx_dw(*args)
    with dw_fp16(False):
        hilo = moe.bwd_dx_dw(*args)
    assert moe.device_error() == 0
    _oracle_check(inp, f16, wd_host=to_host(wd))
    others = [e for e in heavy if e != big]
    for i in (1, 2):
        a, b = to_host(f16[i]), to_host(hilo[i])
        assert _flipped(a[big], b[big]) < 0.01, "the overflowing expert kept the fp16 pass"
        assert min(_flipped(a[e], b[e]) for e in others) > 0.01, "another heavy expert lost the fp16 pass"
    for name, i in (("dX", 0), ("d_logits", 3)):
        assert torch.equal(f16[i], hilo[i]), name
