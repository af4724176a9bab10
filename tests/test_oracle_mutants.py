"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a temporary copy of the oracle source (never
in the real one), compiles it on the CPU, and runs the pin battery of
test_oracle_route / _dispatch / _layer / _activations / _router against it: at least one pin must fail.
"""
import os
import shutil

import pytest

import oracle
from tests import test_oracle_activations as P_A
from tests import test_oracle_dispatch as P_D
from tests import test_oracle_layer as P_L
from tests import test_oracle_route as P_R
from tests import test_oracle_router as P_RP

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.cpp")

MUTANTS = {
    "tie_break_reversed": ("return ia < ib;", "return ia > ib;"),
    "nan_ranked_first": ("if (na != nb) return nb;", "if (na != nb) return na;"),
    "softmax_drops_first_term": ("for (int j = 0; j < k; ++j) {\n      ex[j] = std::exp(l[order[j]] - m);\n      s += ex[j];",
                                 "for (int j = 0; j < k; ++j) {\n      ex[j] = std::exp(l[order[j]] - m);\n      if (j) s += ex[j];"),
    "dispatch_not_stable": ("for (long long s = 0; s < R; ++s) {\n    int e = ids[s];",
                            "for (long long s = R - 1; s >= 0; --s) {\n    int e = ids[s];"),
    "gate_up_rows_swapped": ("const uint16_t* wg = wgu_e + static_cast<size_t>(n) * H;\n    const uint16_t* wu = gated(act) ? wgu_e + static_cast<size_t>(I + n) * H : nullptr;",
                             "const uint16_t* wu = wgu_e + static_cast<size_t>(n) * H;\n    const uint16_t* wg = wgu_e + static_cast<size_t>(I + n) * H;"),
    "silu_sign": ("inline float silu(float a) { return a / (1.0f + std::exp(-a)); }",
                  "inline float silu(float a) { return a / (1.0f + std::exp(a)); }"),
    "down_transposed": ("for (int n = 0; n < I; ++n) a += hq[n] * bf16_to_float(wr[n]);",
                        "for (int n = 0; n < I; ++n) a += hq[n] * bf16_to_float(wd_e[static_cast<size_t>(n) * H + c]);"),
    "combine_weight_dropped": ("acc[c] += round_to_bf16(wj * o[c]);", "acc[c] += round_to_bf16(o[c]);"),
    "grouped_weight_dropped": ("float_to_bf16(w_perm[r] * o[c]);", "float_to_bf16(o[c]);"),
    "swiglu_grad_sign": ("dg[n] = ((dh * u[n]) * s) * (1.0f + g[n] * (1.0f - s));",
                         "dg[n] = ((dh * u[n]) * s) * (1.0f - g[n] * (1.0f - s));"),
    "dx_up_term_dropped": ("          if (wu) acc[h] += du[n] * bf16_to_float(wu[h]);\n", ""),
    "router_grad_sign": ("dl[ids[static_cast<size_t>(t) * k + j]] = wj * (gam[j] - S);",
                         "dl[ids[static_cast<size_t>(t) * k + j]] = wj * (gam[j] + S);"),
    "router_grad_unweighted_gamma": ("for (int j = 0; j < k; ++j) S += w[static_cast<size_t>(t) * k + j] * gam[j];",
                                     "for (int j = 0; j < k; ++j) S += gam[j];"),
    "dwd_weight_dropped": ("float wdy = wj * bf16_to_float(dyr[c]);", "float wdy = bf16_to_float(dyr[c]);"),
    "dwgu_wrong_input_row": ("const uint16_t* xr = x + static_cast<size_t>(rws[r].t) * H;",
                             "const uint16_t* xr = dy + static_cast<size_t>(rws[r].t) * H;"),
    "dhu_reads_gate_weights": ("const uint16_t* wr = wd_e + static_cast<size_t>(c) * I;\n    for (int n = 0; n < I; ++n) dHu[n]",
                               "const uint16_t* wr = wd_e + static_cast<size_t>(c) * I + 1;\n    for (int n = 0; n < I - 1; ++n) dHu[n]"),
}


def _battery():
    """Every pin that can be run as a plain call, on the current oracle build."""
    P_R.test_ids_match_bruteforce_sort(50, 37, 5, True)
    P_R.test_weights_are_renormalised_softmax(40, 64, 6)
    P_R.test_nan_logits_rank_last_and_ids_distinct()
    P_R.test_closed_form_worked_example()
    P_D.test_matches_stable_argsort(300, 37, 5, 0.3)
    for wl in (P_L.TINY, P_L.RAGGED, P_L.ZIPF):
        P_L.test_forward_matches_fp64_dense(wl)
        P_L.test_forward_is_dispatch_grouped_combine(wl)
        P_L.test_backward_matches_fp64_autograd(wl)
    P_L.test_router_gradient_by_central_differences()
    P_L.test_weight_gradient_by_central_differences()
    P_L.test_identity_expert_roundtrip()
    P_L.test_closed_form_worked_example()


# Mistakes in the gated-activation variants, caught by the activation pins.
ACT_MUTANTS = {
    "oai_alpha": ("constexpr float kOaiAlpha = 1.702f;", "constexpr float kOaiAlpha = 1.0f;"),
    "oai_plus_one_dropped": ("return (gc * sigmoid(kOaiAlpha * gc)) * (uc + 1.0f);",
                             "return (gc * sigmoid(kOaiAlpha * gc)) * uc;"),
    "bounded_up_unclamped": ("return silu(gc) * uc;", "return silu(gc) * u;"),
    "bounded_gate_grad_not_blocked": ("*dhdg = (g <= c) ? uc * s * (1.0f + gc * (1.0f - s)) : 0.0f;",
                                      "*dhdg = uc * s * (1.0f + gc * (1.0f - s));"),
    "gelu_cubic_term_dropped": ("constexpr float kGeluK1 = 0.044715f;", "constexpr float kGeluK1 = 0.0f;"),
    "geglu_grad_second_term_dropped": ("const float dgelu = 0.5f * (1.0f + t) + 0.5f * g * (1.0f - t * t) * kGeluK0 * (1.0f + 3.0f * kGeluK1 * g * g);",
                                       "const float dgelu = 0.5f * (1.0f + t);"),
    "reglu_grad_not_gated": ("*dhdg = (g > 0.0f) ? u : 0.0f;", "*dhdg = u;"),
    "relu2_not_squared": ("      return r * r;\n", "      return r;\n"),
    "relu2_grad_halved": ("*dhdg = 2.0f * std::max(g, 0.0f);", "*dhdg = std::max(g, 0.0f);"),
    "relu2_grad_not_gated": ("*dhdg = 2.0f * std::max(g, 0.0f);", "*dhdg = 2.0f * g;"),
}


def _act_battery():
    for act, clamp in P_A.VARIANTS:
        P_A.test_forward_matches_fp64_dense(act, clamp)
        P_A.test_backward_matches_fp64_autograd(act, clamp)
    for case in P_A.CLOSED_FORM:
        P_A.test_closed_form_values(*case)


def test_battery_passes_on_the_real_oracle():
    _battery()
    _act_battery()
    _router_battery()


# Mistakes in the router projection and its backward, caught by the router pins.
ROUTER_MUTANTS = {
    "router_bias_dropped": ("logits[static_cast<size_t>(t) * E + e] = bias ? acc + bias[e] : acc;",
                            "logits[static_cast<size_t>(t) * E + e] = acc;"),
    "router_logits_sum_short": ("for (int h = 0; h < H; ++h) acc += bf16_to_float(xr[h]) * bf16_to_float(we[h]);",
                                "for (int h = 0; h < H - 1; ++h) acc += bf16_to_float(xr[h]) * bf16_to_float(we[h]);"),
    "router_dx_in_dropped": ("const float base = dx_in ? bf16_to_float(dx_in[static_cast<size_t>(t) * H + h]) : 0.0f;",
                             "const float base = 0.0f;"),
    "router_dx_weight_transposed": ("for (int h = 0; h < H; ++h) acc[h] += dl[e] * bf16_to_float(we[h]);",
                                    "for (int h = 0; h < H; ++h) acc[h] += dl[e] * bf16_to_float(wr[static_cast<size_t>(h) * E + e]);"),
    "router_dwr_wrong_operand": ("for (int h = 0; h < H; ++h) acc[h] += d * bf16_to_float(xr[h]);",
                                 "for (int h = 0; h < H; ++h) acc[h] += d * bf16_to_float(wr[static_cast<size_t>(e) * H + h]);"),
    "router_dbias_sign": ("        db += d;\n", "        db -= d;\n"),
}


def _router_battery():
    for shape in P_RP.SHAPES:
        P_RP.test_logits_match_fp64_within_summation_bound(*shape, True)
        P_RP.test_backward_matches_fp64_autograd_dense(*shape, True)
    P_RP.test_logits_equal_the_input_recipe_sum()
    P_RP.test_closed_form_values()
    for wl in P_RP.LAYERS:
        P_RP.test_layer_with_router_matches_fp64_autograd(wl)
    P_RP.test_top1_routing_gives_no_router_gradient()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / "mutant.cpp"
    path.write_text(src.replace(before, after))
    lib = oracle.open_library(oracle.compile_source(str(path), str(tmp_path / "libmutant.so")))
    with oracle.using(lib):
        with pytest.raises((AssertionError, ValueError)):
            _battery()
    shutil.rmtree(tmp_path, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(ACT_MUTANTS))
def test_planted_activation_mistake_is_caught(name, tmp_path):
    before, after = ACT_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / "mutant.cpp"
    path.write_text(src.replace(before, after))
    lib = oracle.open_library(oracle.compile_source(str(path), str(tmp_path / "libmutant.so")))
    with oracle.using(lib):
        with pytest.raises((AssertionError, ValueError)):
            _act_battery()
    shutil.rmtree(tmp_path, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(ROUTER_MUTANTS))
def test_planted_router_mistake_is_caught(name, tmp_path):
    before, after = ROUTER_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / "mutant.cpp"
    path.write_text(src.replace(before, after))
    lib = oracle.open_library(oracle.compile_source(str(path), str(tmp_path / "libmutant.so")))
    with oracle.using(lib):
        with pytest.raises((AssertionError, ValueError)):
            _router_battery()
    shutil.rmtree(tmp_path, ignore_errors=True)
