"""bench.py's host-side bookkeeping, on CPU.

Every rate and roofline fraction in the bench line divides by these numbers: the flops credited
to a step and to each GEMM, the minimum bytes of each kernel, the peaks, and the gate that keeps
a stale DRAM-traffic capture out of the line.  They are pinned here against their closed forms
(the expert MLP's 6 R H I forward and 12 R H I backward multiply-add flops, with R = T k rows).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synthetic  # noqa: E402

BENCH = synthetic.workload("fwd_T8192_H2048_I512_E256_k8")
FWD_GEMMS = ("gemm_gate_up_swiglu", "gemm_down_scale")
BWD_GEMMS = ("gemm_bwd_dh", "gemm_bwd_dx", "gemm_bwd_dw_gate_up", "gemm_bwd_dw_down")


def test_step_flops_are_18_RHI_for_gated_experts():
    R, H, I = BENCH.R, BENCH.H, BENCH.I
    fl = bench.step_flops(BENCH)
    assert (fl["fwd"], fl["bwd"], fl["total"]) == (6 * R * H * I, 12 * R * H * I, 18 * R * H * I)
    assert fl["total"] == 1_236_950_581_248  # 65536 rows x 2048 x 512


def test_two_weight_experts_and_the_router_projection():
    T, H, I, E, R = BENCH.T, BENCH.H, BENCH.I, BENCH.E, BENCH.R
    assert bench.step_flops(BENCH, gated=False)["total"] == 12 * R * H * I
    fr = bench.step_flops(BENCH, router=True)
    assert fr["fwd"] - 6 * R * H * I == 2 * T * H * E   # x Wr^T
    assert fr["bwd"] - 12 * R * H * I == 4 * R * H      # its dX and dWr over the selected pairs


@pytest.mark.parametrize("gated", [True, False])
def test_the_gemms_account_for_the_whole_step(gated):
    up = "gemm_gate_up_swiglu" if gated else "gemm_up_relu2"
    fwd = sum(bench.kernel_work(BENCH, n, gated)[1] for n in (up, "gemm_down_scale"))
    bwd = sum(bench.kernel_work(BENCH, n, gated)[1] for n in BWD_GEMMS)
    fl = bench.step_flops(BENCH, gated)
    assert (fwd, bwd) == (fl["fwd"], fl["bwd"])
    assert all(bench.kernel_work(BENCH, n, gated)[0] == "flop" for n in FWD_GEMMS + BWD_GEMMS)


def test_dw_gate_up_minimum_bytes():
    H, I, E, R = BENCH.H, BENCH.I, BENCH.E, BENCH.R
    # dgu [R, 2I] and x_perm [R, H] read once, dW_gate_up [E, 2I, H] written once, all bf16
    expect = R * 2 * I * 2 + R * H * 2 + E * 2 * I * H * 2
    assert bench.gemm_bytes(BENCH, "gemm_bwd_dw_gate_up", experts_used=E) == expect == 1_476_395_008


def test_forward_weight_bytes_count_only_experts_with_rows():
    H, I = BENCH.H, BENCH.I
    full = bench.gemm_bytes(BENCH, "gemm_gate_up_swiglu", experts_used=256)
    half = bench.gemm_bytes(BENCH, "gemm_gate_up_swiglu", experts_used=128)
    assert full - half == 128 * 2 * I * H * 2


def test_row_copy_bytes():
    T, H, R = BENCH.T, BENCH.H, BENCH.R
    assert bench.kernel_work(BENCH, "gather_rows") == ("byte", T * H * 2 + R * H * 2 + R * 4)
    assert bench.kernel_work(BENCH, "combine") == ("byte", R * H * 2 + T * H * 2 + R * 4)
    assert bench.kernel_work(BENCH, "no_such_kernel") == ("byte", 0)


def test_peaks_come_from_the_measured_file_or_the_stated_fallback(tmp_path, monkeypatch):
    p = bench.load_peaks()
    assert p["hbm_gbs"] > 0 and p["bf16_tflops"] >= p["bf16_tflops_sustained"] > 0
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))  # no peaks file there
    assert bench.load_peaks() == dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                                      source="fallback")


def test_traffic_is_reported_only_for_the_kernel_source_it_was_taken_on(monkeypatch):
    import json

    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        entry = json.load(f)[BENCH.name]["gemm_bwd_dw_gate_up"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: entry["kernel_source_sha256"])
    assert bench.load_traffic(BENCH.name, "gemm_bwd_dw_gate_up") == entry["dram_bytes_per_launch"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 64)
    assert bench.load_traffic(BENCH.name, "gemm_bwd_dw_gate_up") is None
    assert bench.load_traffic("no_such_workload", "gemm_bwd_dw_gate_up") is None


def test_defaults_are_one_gpu_and_the_largest_workload(monkeypatch):
    """The default line is the largest single-GPU workload (the most flops per step of the five)."""
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse_args()
    largest = max(synthetic.WORKLOADS.values(), key=lambda w: bench.step_flops(w)["total"])
    assert (a.gpus, a.impl, a.workload, a.inputs, a.act) == (1, "ours", largest.name, "x_perm", "swiglu")
    assert largest.name == "fwd_zipf_T8192_H4096_I1024_E512_k10"
    assert a.warmup >= 3 and a.steps >= 1 and not a.router and not a.no_train_shape
    assert synthetic.workload(bench.TRAIN_SHAPE).as_dict() == dict(workload=bench.TRAIN_SHAPE, T=8192, H=2048, I=768,
                                                                   E=128, k=8)


def test_fp16_pass_rows_follow_the_library_rule():
    counts = [383, 384, 1000, 0, 5]
    assert bench.f16_pass_rows(counts, 32768, True, True) == 1384
    assert bench.f16_pass_rows(counts, 32767, True, True) == 0   # batch below 32768 routed rows
    assert bench.f16_pass_rows(counts, 65536, False, True) == 0  # two-weight experts
    assert bench.f16_pass_rows(counts, 65536, True, False) == 0  # token-major (gathered) inputs


def test_fp16_row_copy_bytes():
    wl = synthetic.workload("fwd_zipf_T8192_H4096_I1024_E512_k10")
    T, H, R = wl.T, wl.H, wl.R
    plain = bench.kernel_work(wl, "gather_rows")[1]
    assert bench.kernel_work(wl, "gather_rows_f16", f16_rows=0)[1] == plain
    assert bench.kernel_work(wl, "f16_prep", f16_rows=0)[1] == 0
    f16_rows = 40000
    # on top of the plain dY copy: one x row per token read, fp16 dY and x rows written for the heavy experts
    extra = bench.kernel_work(wl, "gather_rows_f16", f16_rows=f16_rows)[1] - plain
    assert extra == T * H * 2 + 2 * f16_rows * H * 2
    assert bench.kernel_work(wl, "f16_prep", f16_rows=f16_rows)[1] >= 2 * T * H * 2  # |x| and |dY| maxima read
