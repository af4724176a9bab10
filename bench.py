#!/usr/bin/env python3
"""Throughput of the routed MoE layer (forward + backward) on GB300.

One step = the whole layer on one batch: router top-k, dispatch, grouped
SwiGLU expert GEMMs, combine, and the backward (dX, dW_gate_up, dW_down,
d_logits), all through the C-ABI library.  Inputs are seeded synthetic data
with the workload's shapes (no dataset).  The printed JSON line carries:

* value         fwd+bwd algorithmic TFLOP/s (18 * T*k * H * I flop per step), all ranks
* roofline      the dominant kernel's algorithmic FLOP/s (or bytes/s) over its mean
                device duration, from the library's per-launch CUDA-event trace
* e2e           the same metric with host buffers: pinned host->device copies of the
                step's inputs and device->host copies of its outputs inside the timed loop
* cpu_baseline  the CPU oracle on a bounded sample of the same workload
* clocks        SM clock / throttle reasons sampled with nvidia-smi during the timed loop
* inference_forward  the forward alone without saved derivative factors (nothing kept for a
                backward): ms, TFLOP/s, and each expert GEMM's TFLOP/s against the bf16 peaks
* sustained     the same step graph replayed back to back for at least a second, with the
                median SM clock of that window (the power cap settles in over such a run)
* train_shape_forward  the training shape (H=2048, I=768, E=128, top-8, 8192 tokens), the one
                shape whose forward expert GEMMs are tensor-bound: each GEMM's TFLOP/s in its
                training step and in an inference forward, against the burst and sustained
                bf16 peaks, with the clocks sampled over those replays

``--impl reference`` times the CPU oracle itself on the host cores (the only
reference implementation of this method that exists here).
Multi-GPU: the layer has no exchange step on one GPU's data path, so N ranks
run N independent replicas (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE layer fwd/bwd TFLOP/s and tokens/s on 1 GB300; % of BF16 tensor-core peak"
# The largest single-GPU workload: the 4096/1024/512-expert top-10 model shape with Zipf(1.2)-skewed
# expert load.  The training shape's forward GEMMs get their own record (train_shape_forward).
DEFAULT_WORKLOAD = "fwd_zipf_T8192_H4096_I1024_E512_k10"
TRAIN_SHAPE = "train_T8192_H2048_I768_E128_k8"
L2_BYTES = 129 * 2 ** 20


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-train-shape", action="store_true", help="leave out the training shape's forward-GEMM record")
    ap.add_argument("--no-graph", action="store_true", help="launch the timed steps one by one instead of "
                    "replaying them as one captured CUDA graph")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU work of the oracle baseline sample")
    ap.add_argument("--inputs", choices=["x_perm", "gather"], default="x_perm",
                    help="expert GEMM inputs: expert-major copies (x_perm, dy_perm) read as dense tiles, or the "
                    "memory-lean path that gathers x and dY rows by token inside the GEMMs")
    ap.add_argument("--act", choices=["swiglu", "swiglu_bounded", "swiglu_oai", "geglu", "reglu", "relu2"],
                    default="swiglu", help="activation of the expert MLP (x_perm inputs only for the others; relu2 "
                    "runs two-weight experts whose up weight is the gate half of the synthetic W_gu)")
    ap.add_argument("--act-clamp", type=float, default=7.0, help="clamp of swiglu_bounded / limit of swiglu_oai")
    ap.add_argument("--router", action="store_true", help="start the step from x: the router projection "
                    "logits = x Wr^T (+ bias) runs on the GPU, and its backward adds the router's dX and gives "
                    "dWr, dbias (default: the logits are the layer's input)")
    args = ap.parse_args()
    if args.act != "swiglu" and args.inputs == "gather":
        ap.error("--act other than swiglu runs on x_perm inputs")
    return args


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# ---------------------------------------------------------------- algorithmic work
def step_flops(wl, gated: bool = True, router: bool = False) -> dict:
    """Gated experts: gate/up 4 + down 2 forward; dH 2 + dX 4 + dW_gu 4 + dW_d 2 backward (x R H I).
    Two-weight (relu2) experts: up 2 + down 2; dH 2 + dX 2 + dW_up 2 + dW_d 2.
    With the router projection: 2 T H E forward (x Wr^T); 4 R H backward (its dX and dWr, each one
    multiply-add per selected (token, expert) pair and column: d_logits vanish off the top-k)."""
    rhi = wl.R * wl.H * wl.I
    fwd, bwd = (6, 12) if gated else (4, 8)
    fwd, bwd = fwd * rhi, bwd * rhi
    if router:
        fwd += 2 * wl.T * wl.H * wl.E
        bwd += 4 * wl.R * wl.H
    return dict(fwd=fwd, bwd=bwd, total=fwd + bwd)


def gemm_bytes(wl, name: str, experts_used: int, gated: bool = True) -> int:
    """Minimum DRAM bytes of one grouped-GEMM launch: every operand read once and every output
    written once, at its algorithmic precision (bf16 activations and weights, the fp32 SwiGLU
    derivative factors the forward saves; the hi/lo second halves of the weight-gradient
    operands are an implementation choice and are not counted).  Weights count only for
    experts that received rows.  nin = rows of the first weight per expert (2I gated, I relu2)."""
    H, I, E, R = wl.H, wl.I, wl.E, wl.R
    nin = 2 * I if gated else I
    w_gu = experts_used * nin * H * 2
    w_d = experts_used * H * I * 2
    act_h, act_x = R * H * 2, R * I * 2  # [R, H] and [R, I] bf16
    dgu = R * nin * 2
    factors = R * nin * 4
    up = act_h + w_gu + act_x + factors  # x_perm, W_gu -> h, factors
    return {
        "gemm_gate_up_swiglu": up, "gemm_gate_up_glu": up, "gemm_up_relu2": up,
        "gemm_down_scale": act_x + w_d + act_h,                   # h, W_d -> y_perm
        "gemm_bwd_dh": act_h + w_d + factors + act_x + dgu + act_x,  # dY rows, W_d, factors, h -> dgu, w h
        "gemm_bwd_dx": dgu + w_gu + act_h,                        # dgu, W_gu -> dx_perm
        "gemm_bwd_dw_gate_up": dgu + act_h + E * nin * H * 2,     # dgu, x_perm -> dW_gate_up (all experts)
        "gemm_bwd_dw_down": act_h + act_x + E * H * I * 2,         # dY rows, w h -> dW_down (all experts)
        "gemm_router_logits": wl.T * H * 2 + E * H * 2 + wl.T * E * 4,  # x, Wr -> logits (fp32)
    }[name]


def f16_pass_rows(counts, R: int, gated: bool, expert_major: bool) -> int:
    """Routed rows of the experts that take the backward's fp16 weight-gradient pass, by the
    library's rule: gated experts, expert-major inputs, a batch of at least 32768 routed rows, and
    experts with at least 384 rows each.  0 when the pass does not apply."""
    if not (gated and expert_major and R >= 32768):
        return 0
    return sum(int(c) for c in counts if c >= 384)


def kernel_work(wl, name: str, gated: bool = True, f16_rows: int = 0):
    """(kind, algorithmic amount per launch): kind 'flop' for GEMMs, 'byte' for the rest.  f16_rows:
    routed rows of the experts that take the backward's fp16 weight-gradient pass (at least 384 rows
    each; 0: none), whose dY and x rows the row copy also writes as fp16, after the largest |dY|, |x|
    are read."""
    T, H, I, E, k, R = wl.T, wl.H, wl.I, wl.E, wl.k, wl.R
    rhi = R * H * I
    nunits = math.ceil(R / 256)
    g = 2 if gated else 1  # rows of the first weight per expert, in units of I
    gemm = {"gemm_gate_up_swiglu": 4 * rhi, "gemm_gate_up_glu": 4 * rhi, "gemm_up_relu2": 2 * rhi,
            "gemm_down_scale": 2 * rhi, "gemm_bwd_dh": 2 * rhi,
            "gemm_bwd_dx": 2 * g * rhi, "gemm_bwd_dw_gate_up": 2 * g * rhi, "gemm_bwd_dw_down": 2 * rhi,
            "gemm_router_logits": 2 * T * H * E}
    if name in gemm:
        return "flop", gemm[name]
    nbytes = {
        "route_topk": T * E * 4 + T * k * 8,
        "dispatch_hist": R * 4 + nunits * E * 4,
        "dispatch_scan": 2 * nunits * E * 4 + E * 4,
        "dispatch_scatter": R * 4 * 5 + nunits * E * 4,
        "dispatch_small": R * 4 * 5 + (2 * E + 1) * 4,  # ids, w read; both maps, w_perm written; counts, m_indptr
        "gather_rows": T * H * 2 + R * H * 2 + R * 4,
        # dY (and, for the fp16 copies, one x row per token) read; dy_perm (and dy16, x16) written
        "gather_rows_f16": (2 * T * H * 2 + R * H * 2 + 2 * f16_rows * H * 2 + R * 4) if f16_rows
                           else (T * H * 2 + R * H * 2 + R * 4),
        "f16_prep": (2 * T * H * 2 + T * 4) if f16_rows else 0,
        "combine": R * H * 2 + T * H * 2 + R * 4,
        "router_grad": T * E * 4 + R * (4 * math.ceil(I / 256) + 12),
        "tile_schedule": (E + 1) * 8,
        "router_dx": 2 * T * H * 2 + E * H * 2 + T * k * 8,        # dX read + written, Wr, ids + d_logits
        "router_dw": T * H * 2 + E * H * 2 + R * 8 + E * 8,         # x, dWr, row_to_slot + d_logits, m_indptr
    }
    return "byte", nbytes.get(name, 0)


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.seek(0)
        rows = [l.strip().split(", ") for l in self.file.read().splitlines() if l.strip()]
        sm, mx, pw, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                pw.append(float(r[3]))
            except (ValueError, IndexError):
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [s for s, p in zip(sm, pw) if p >= 0.5 * max(pw)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(pw)}


def gpu_index_for(local_rank: int) -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


# ---------------------------------------------------------------- CPU oracle (baseline / reference arm)
def oracle_sample(wl, inp, ids, w, n_tokens: int, experts, act=("swiglu", 0.0), router=False) -> float:
    """Runs the oracle's fwd + bwd on n_tokens tokens and dW on `experts` (with `router`, also the
    router projection of those tokens and its backward); returns algorithmic flop."""
    import numpy as np

    import oracle

    toks = np.arange(n_tokens, dtype=np.int32)
    kw = dict(act=act[0], clamp=act[1])
    if router:
        oracle.router_logits(inp["x"][:n_tokens], inp["wr"], inp["bias"])
    oracle.forward_tokens(inp["x"], inp["wgu"], inp["wd"], ids, w, toks=toks, **kw)
    dx, dl = oracle.backward_tokens(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w, toks=toks, **kw)
    g = 1 if act[0] == "relu2" else 2  # rows of the first weight per expert, in units of I
    flop = (2 * g + 2 + 2 + 2 * g) * n_tokens * wl.k * wl.H * wl.I  # fwd + dH + dX per routed row
    if router:
        oracle.router_backward(dl, inp["x"][:n_tokens], inp["wr"], dx)
        flop += 2 * n_tokens * wl.H * wl.E + 4 * n_tokens * wl.k * wl.H
    if len(experts):
        oracle.backward_dw(inp["x"], inp["dy"], inp["wgu"], inp["wd"], ids, w,
                           experts=np.asarray(experts, dtype=np.int32), **kw)
        rows = np.bincount(ids.ravel(), minlength=wl.E)[np.asarray(experts)].sum()
        flop += (2 * g + 2) * int(rows) * wl.H * wl.I
    return float(flop)


def size_oracle_sample(wl, inp, ids, w, seconds: float, act=("swiglu", 0.0), router=False):
    """Tokens / experts for a sample of about `seconds` of oracle work (one calibration call)."""
    import numpy as np

    import oracle

    n_cal = min(wl.T, 2 * oracle.default_threads())  # enough tokens to engage every thread
    t0 = time.perf_counter()
    oracle_sample(wl, inp, ids, w, n_cal, [], act, router)
    per_tok = max((time.perf_counter() - t0) / n_cal, 1e-6)
    n_tok = int(max(1, min(wl.T, seconds * 0.7 / per_tok)))
    # dW runs one expert per thread: up to `threads` mid-size experts whose largest row count
    # keeps one thread's share near 30 % of the budget (a row costs about 1.5 token-rows of work)
    threads = oracle.default_threads()
    per_row_single = per_tok * threads / wl.k * 1.5
    counts = np.bincount(ids.ravel(), minlength=wl.E)
    order = [int(e) for e in np.argsort(counts, kind="stable") if counts[e] > 0]
    mid = order[len(order) // 2:] + order[: len(order) // 2][::-1]
    experts = [e for e in mid if counts[e] * per_row_single <= 0.3 * seconds][:threads]
    return n_tok, experts


def run_reference(args, rank, world):
    if rank != 0:
        return
    import numpy as np

    import oracle
    import synthetic

    wl = synthetic.workload(args.workload)
    inp = synthetic.make_inputs(wl, seed=args.seed, want=("x", "logits", "wgu", "wd", "dy", "wr"))
    if args.act == "relu2":  # two-weight experts: the up weight is the gate half of W_gu
        inp["wgu"] = np.ascontiguousarray(inp["wgu"][:, : wl.I])
    ids, w = oracle.route_topk(inp["logits"], wl.k)
    total_steps = args.warmup + args.steps
    per_step = max(0.05, min(5.0, 150.0 / max(total_steps, 1)))
    n_tok, _ = size_oracle_sample(wl, inp, ids, w, per_step, (args.act, args.act_clamp), args.router)
    counts = np.bincount(ids.ravel(), minlength=wl.E)
    nonempty = [int(e) for e in np.nonzero(counts)[0]]
    flops = []
    times = []
    for i in range(total_steps):
        experts = [nonempty[i % len(nonempty)]] if nonempty else []
        t0 = time.perf_counter()
        f = oracle_sample(wl, inp, ids, w, n_tok, experts, (args.act, args.act_clamp), args.router)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            flops.append(f)
            times.append(dt)
    value = sum(flops) / sum(times) / 1e12
    cores = oracle.default_threads()
    sample = (f"{n_tok} of {wl.T} tokens (forward + dX + d_logits"
              f"{', router projection and its backward' if args.router else ''}) and one expert's dW per step, "
              f"oracle threads={cores}")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": dict(wl.as_dict(), pass_="forward+backward"),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    line["config"]["pass"] = line["config"].pop("pass_")
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- ranks
# N GPUs run N independent replicas of the layer step (the path has no exchange step on one
# GPU's data).  The ranks meet only around the timed region: a barrier on both sides, the
# slowest rank's time, and the whole-job rate from it.
def rank_barrier(dist) -> None:
    if dist is not None:
        dist.barrier()


def rank_max(v: float, dist, device) -> float:
    """The largest `v` over all ranks (`device`: where the reduction tensor lives for the backend)."""
    if dist is None:
        return v
    import torch

    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_rank: float, slowest_ms: float) -> float:
    """Units per second of the whole job: every rank processed `units_per_rank` within `slowest_ms`."""
    return world * units_per_rank / (slowest_ms * 1e-3)


# ---------------------------------------------------------------- our arm
class Layer:
    """Device buffers and the layer calls of one workload (forward, backward, one step)."""

    def __init__(self, args, wl, dev, inp, act="swiglu", inputs="x_perm", router=False):
        import numpy as np
        import torch

        import mixture_experts_routed_router_gb300 as moe

        self.wl, self.dev = wl, dev
        T, H, I, E, k, R = wl.T, wl.H, wl.I, wl.E, wl.k, wl.R
        self.gated = gated = act != "relu2"
        if not gated:  # two-weight experts: the up weight W_up [E, I, H] is the gate half of W_gu
            inp["wgu"] = np.ascontiguousarray(inp["wgu"][:, :I])
        nin = 2 * I if gated else I  # rows of the first weight per expert

        def to_dev(a):
            a = np.ascontiguousarray(a)
            if a.dtype == np.uint16:
                return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
            return torch.from_numpy(a).to(dev)

        self.logits, self.x, self.dy = to_dev(inp["logits"]), to_dev(inp["x"]), to_dev(inp["dy"])
        wgu, wd = to_dev(inp["wgu"]), to_dev(inp["wd"])
        self.weight_bytes = (wgu.numel() + wd.numel()) * 2
        bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
        e = lambda *s, dt=bf: torch.empty(s, dtype=dt, device=dev)
        self.empty = e
        ids, w = e(T, k, dt=i32), e(T, k, dt=f32)
        dbuf = dict(counts=e(E, dt=i32), m_indptr=e(E + 1, dt=i32), row_to_slot=e(R, dt=i32),
                    slot_to_row=e(R, dt=i32), w_perm=e(R, dt=f32))
        gather = inputs == "gather"
        if not gather:
            dbuf["x_perm"] = e(R, H)
        fbuf = dict(h_perm=e(R, I), gu_perm=e(R, nin, dt=f32), y_perm=e(R, H))
        self.Y = Y = e(T, H)
        bbuf = dict(dx=e(T, H), dw_gate_up=e(E, nin, H), dw_down=e(E, H, I), d_logits=e(T, E, dt=f32))
        ws_d = e(moe.workspace_bytes("dispatch", T=T, E=E, k=k), dt=torch.uint8)
        ws_f = e(moe.workspace_bytes("grouped_swiglu_fwd", R=R, H=H, I=I, E=E), dt=torch.uint8)
        ws_b = e(moe.workspace_bytes("bwd_dx_dw", T=T, H=H, I=I, E=E, k=k, saved_gu=True, gather=gather),
                 dt=torch.uint8)
        self.dbuf = dbuf
        # router: the router projection (weights resident like the experts'); with it the step's input
        # is x alone and the logits buffer is an output of the step
        wr = to_dev(inp["wr"]) if router else None
        rbias = to_dev(inp["bias"]) if router and inp["bias"] is not None else None
        rbuf = dict(dw_router=e(E, H), d_bias=e(E, dt=f32)) if router else None

        # inputs x_perm (default): the dispatch writes the expert-major copy x_perm (and the backward
        # its dy_perm), which the GEMMs read as dense TMA tiles.  inputs gather: the layer on
        # token-major x and dY, the expert GEMMs copying their rows by token, so no expert-major copy
        # exists (less memory, slower).
        # save=False: an inference forward, which keeps no derivative factors for a backward
        def forward(lg, xx, y_out=None, save=True):
            if router:
                moe.router_logits(xx, wr, rbias, out=lg)
            moe.route_topk(lg, k, topk_ids=ids, topk_w=w)
            moe.dispatch(ids, w, None if gather else xx, E, out=dbuf, workspace=ws_d)
            if gather:
                moe.grouped_swiglu_fwd_gather(xx, dbuf["row_to_slot"], k, dbuf["m_indptr"], wgu, wd, dbuf["w_perm"],
                                              save_gu=save, out=fbuf, workspace=ws_f)
            elif act != "swiglu":
                moe.grouped_glu_fwd(dbuf["x_perm"], dbuf["m_indptr"], wgu, wd, dbuf["w_perm"], act, args.act_clamp,
                                    save_gu=save, out=fbuf, workspace=ws_f)
            else:
                moe.grouped_swiglu_fwd(dbuf["x_perm"], dbuf["m_indptr"], wgu, wd, dbuf["w_perm"], save_gu=save,
                                       out=fbuf, workspace=ws_f)
            moe.combine(fbuf["y_perm"], dbuf["slot_to_row"], T, k, out=Y if y_out is None else y_out)

        def backward(dyy, xx, dx_out=None, dl_out=None):
            out = dict(bbuf)
            if dx_out is not None:
                out.update(dx=dx_out, d_logits=dl_out)
            # the saved derivative factors make the backward the same for every gated activation;
            # two-weight experts (relu2) have their own operand shapes
            args_b = (dyy, xx if gather else dbuf["x_perm"], fbuf["h_perm"], fbuf["gu_perm"], ids, w,
                      dbuf["m_indptr"], dbuf["row_to_slot"], dbuf["slot_to_row"], dbuf["w_perm"], wgu, wd)
            if not gated:
                moe.bwd_dx_dw_glu(*args_b, act, args.act_clamp, out=out, workspace=ws_b)
            else:
                (moe.bwd_dx_dw_gather if gather else moe.bwd_dx_dw)(*args_b, out=out, workspace=ws_b)
            if router:  # adds the router's input gradient to dX; dWr, dbias
                moe.router_bwd(out["d_logits"], ids, dbuf["m_indptr"], dbuf["row_to_slot"], xx, wr, out["dx"],
                               dw_router=rbuf["dw_router"], d_bias=rbuf["d_bias"])

        self.forward, self.backward = forward, backward

    def step(self):
        self.forward(self.logits, self.x)
        self.backward(self.dy, self.x)


def capture(fn, n):
    """One CUDA graph of n calls of fn (the library's calls only enqueue work on the current stream)."""
    import torch

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(n):
            fn()
    return g


def gemm_rates(wl, records, peaks, gated=True) -> dict:
    """Each grouped GEMM's mean duration and TFLOP/s in a trace, against the burst and sustained bf16 peaks."""
    stats = {}
    for name, ms in records:
        s_ = stats.setdefault(name, [0, 0.0])
        s_[0] += 1
        s_[1] += ms
    out = {}
    for name, (n, tot) in sorted(stats.items(), key=lambda kv: -kv[1][1]):
        kind, amount = kernel_work(wl, name, gated)
        if kind != "flop" or tot <= 0:
            continue
        tf = amount / (tot / n * 1e-3) / 1e12
        out[name] = {"avg_us": round(1e3 * tot / n, 2), "tflops": round(tf, 1),
                     "frac_of_bf16_burst": round(tf / peaks["bf16_tflops"], 4),
                     "frac_of_bf16_sustained": round(tf / peaks["bf16_tflops_sustained"], 4)}
    return out


def train_shape_forward(args, dev, local_rank, peaks, max_over_ranks, world) -> dict:
    """The training shape's forward expert GEMMs, in its training step and in an inference forward.

    Each GEMM's rate comes from the library's per-launch trace of a replayed graph (the step's,
    then the inference forward's); the clocks are sampled over both replays."""
    import torch

    import mixture_experts_routed_router_gb300 as moe
    import synthetic

    wl = synthetic.workload(TRAIN_SHAPE)
    inp = synthetic.make_inputs(wl, seed=args.seed, want=("x", "logits", "wgu", "wd", "dy"))
    L = Layer(args, wl, dev, inp)
    for _ in range(3):
        L.step()
    torch.cuda.synchronize()
    n_step, n_fwd = 40, 100
    # The trace logs a record per launch when the graphs are captured; each replay re-times the
    # records' events, so the records read after the last replay hold that replay's durations.
    moe.trace_enable(True)  # stays on until the records are read (turning it off clears them)
    g_step = capture(L.step, n_step)
    n_step_records = moe.load_library().liger_moe_trace_count()  # records of the step graph (not yet timed)
    g_inf = capture(lambda: L.forward(L.logits, L.x, save=False), n_fwd)
    g_step.replay()  # first replays upload the graphs; untimed
    g_inf.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(gpu_index_for(local_rank))
    clocks.start()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    stream = torch.cuda.current_stream()
    ev[0].record(stream)
    g_step.replay()
    ev[1].record(stream)
    ev[2].record(stream)
    g_inf.replay()
    ev[3].record(stream)
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    records = moe.trace_records()
    step_records, inf_records = records[:n_step_records], records[n_step_records:]
    moe.trace_enable(False)
    flags = moe.device_error()
    if flags:
        raise RuntimeError(f"device error flags {flags:#x} in the training-shape record")
    fl = step_flops(wl)
    step_ms = max_over_ranks(ev[0].elapsed_time(ev[1])) / n_step  # traced replays: a few % slower
    inf_ms = max_over_ranks(ev[2].elapsed_time(ev[3])) / n_fwd
    rec = {"workload": wl.name, "config": wl.as_dict(),
           "training_step": {"ms_per_step_traced": round(step_ms, 4),
                             "tflops": round(whole_job_rate(world, fl["total"], step_ms) / 1e12, 2),
                             "gemms": {k_: v for k_, v in gemm_rates(wl, step_records, peaks).items()
                                       if k_ in ("gemm_gate_up_swiglu", "gemm_down_scale")}},
           "inference_forward": {"ms_traced": round(inf_ms, 4),
                                 "tflops": round(whole_job_rate(world, fl["fwd"], inf_ms) / 1e12, 2),
                                 "gemms": gemm_rates(wl, inf_records, peaks)},
           "peaks": {"bf16_burst_tflops": peaks["bf16_tflops"], "bf16_sustained_tflops": peaks["bf16_tflops_sustained"],
                     "source": peaks["source"]},
           "clocks": clock_info,
           "timing": f"library trace of a replayed graph: {n_step} training steps, then {n_fwd} inference forwards"}
    del L, g_step, g_inf
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    import mixture_experts_routed_router_gb300 as moe
    import synthetic

    dist = None
    if world > 1:
        import torch.distributed as dist

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = synthetic.workload(args.workload)
    T, H, I, E, k, R = wl.T, wl.H, wl.I, wl.E, wl.k, wl.R
    inp = synthetic.make_inputs(wl, seed=args.seed, want=("x", "logits", "wgu", "wd", "dy", "wr"))
    L = Layer(args, wl, dev, inp, act=args.act, inputs=args.inputs, router=args.router)
    gated = L.gated
    logits, x, dy, Y, dbuf = L.logits, L.x, L.dy, L.Y, L.dbuf
    forward, backward, step = L.forward, L.backward, L.step
    e = L.empty
    bf, f32 = torch.bfloat16, torch.float32

    def barrier():
        rank_barrier(dist)

    def max_over_ranks(v: float) -> float:
        return rank_max(v, dist, dev)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    flags = moe.device_error()
    if flags:
        raise RuntimeError(f"device error flags {flags:#x} during warm-up")
    experts_used = int((dbuf["counts"] > 0).sum().item())  # experts whose weights the GEMMs read
    f16_rows = f16_pass_rows(dbuf["counts"].cpu().tolist(), wl.R, gated, args.inputs != "gather")

    # ---------------- timed region: K steps, CUDA events on the launching stream
    # The K steps are captured once as a CUDA graph (the library's calls only enqueue work on
    # the current stream) and replayed.  The headline time is an untraced replay.  A second
    # graph of the same K steps, captured with the library's per-launch event trace on (the
    # trace's event records cost a few percent), is replayed right after; its records give
    # the per-kernel durations and the roofline.
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(gpu_index_for(local_rank))
    graph, tgraph, graph_note = None, None, "off (--no-graph): steps launched one by one"
    if not args.no_graph:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for _ in range(args.steps):
                    step()
            moe.trace_enable(True)
            tgraph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(tgraph):
                for _ in range(args.steps):
                    step()
            graph.replay()  # first replays upload the graphs; untimed
            tgraph.replay()
            torch.cuda.synchronize()
            graph_note = f"one CUDA graph of {args.steps} steps (untimed upload replay, then the timed replay)"
        except Exception as exc:  # capture unsupported here: time the steps one by one
            graph, tgraph = None, None
            graph_note = f"capture failed ({type(exc).__name__}): steps launched one by one"
            torch.cuda.synchronize()
    if graph is None:
        moe.trace_enable(True)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for _ in range(args.steps):
            step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    trace_ms = None
    if tgraph is not None:
        ev6, ev7 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev6.record(stream)
        tgraph.replay()
        ev7.record(stream)
        torch.cuda.synchronize()
        trace_ms = ev6.elapsed_time(ev7) / args.steps
    clock_info = clocks.stop()
    records = moe.trace_records()
    launch_counts = moe.trace_launch_counts()
    moe.trace_enable(False)
    elapsed_ms = max_over_ranks(ev0.elapsed_time(ev1))
    flags = moe.device_error()
    if flags:
        raise RuntimeError(f"device error flags {flags:#x} in the timed region")

    fl = step_flops(wl, gated, args.router)
    ms_per_step = elapsed_ms / args.steps
    value = whole_job_rate(world, args.steps * fl["total"], elapsed_ms) / 1e12
    tokens_per_s = whole_job_rate(world, args.steps * T, elapsed_ms)

    # ---------------- sustained: the same untraced step graph replayed back to back for at least
    # a second (the timed region above can be shorter than the time the power cap takes to settle)
    sustained = None
    if graph is not None:
        n_rep = max(1, math.ceil(1200.0 / max(elapsed_ms, 1e-3)))
        sclocks = ClockSampler(gpu_index_for(local_rank))
        sclocks.start()
        barrier()
        torch.cuda.synchronize()
        ev10, ev11 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev10.record(stream)
        for _ in range(n_rep):
            graph.replay()
        ev11.record(stream)
        torch.cuda.synchronize()
        barrier()
        sc = sclocks.stop()
        s_ms = max_over_ranks(ev10.elapsed_time(ev11))
        sustained = {"seconds": round(s_ms / 1e3, 3), "steps": n_rep * args.steps,
                     "ms_per_step": round(s_ms / (n_rep * args.steps), 4),
                     "value": round(whole_job_rate(world, n_rep * args.steps * fl["total"], s_ms) / 1e12, 2),
                     "unit": "TFLOP/s", "sm_mhz_median": sc["sm_mhz"], "clocks": sc}
        flags = moe.device_error()
        if flags:
            raise RuntimeError(f"device error flags {flags:#x} in the sustained replay")

    # forward-only timing (same buffers, launched the same way), for the fwd / bwd split
    ev2, ev3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nf = max(3, args.steps // 2)
    gf = None
    if graph is not None:
        gf = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gf):
            for _ in range(nf):
                forward(logits, x)
        gf.replay()
    torch.cuda.synchronize()
    ev2.record(stream)
    if gf is not None:
        gf.replay()
    else:
        for _ in range(nf):
            forward(logits, x)
    ev3.record(stream)
    torch.cuda.synchronize()
    fwd_ms = max_over_ranks(ev2.elapsed_time(ev3)) / nf

    # inference forward (no derivative factors saved), timed the same way; a traced replay of
    # the same launches gives each expert GEMM's rate
    gi, ti = None, None
    if graph is not None:
        gi = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gi):
            for _ in range(nf):
                forward(logits, x, save=False)
        moe.trace_enable(True)  # stays on until the records are read (turning it off clears them)
        ti = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ti):
            for _ in range(nf):
                forward(logits, x, save=False)
        gi.replay()
        ti.replay()
    torch.cuda.synchronize()
    ev8, ev9 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev8.record(stream)
    if gi is not None:
        gi.replay()
    else:
        for _ in range(nf):
            forward(logits, x, save=False)
    ev9.record(stream)
    torch.cuda.synchronize()
    inf_ms = max_over_ranks(ev8.elapsed_time(ev9)) / nf
    if ti is not None:
        ti.replay()
    else:
        moe.trace_enable(True)
        for _ in range(nf):
            forward(logits, x, save=False)
    torch.cuda.synchronize()
    inf_records = moe.trace_records()
    moe.trace_enable(False)

    # ---------------- per-kernel statistics from the trace of the timed region
    peaks = load_peaks()
    stats = {}
    for name, ms in records:
        s = stats.setdefault(name, [0, 0.0])
        s[0] += 1
        s[1] += ms
    total_kernel_ms = sum(v[1] for v in stats.values()) or 1.0
    kernels = {}
    # a GEMM is HBM-bound when its algorithmic intensity is below the ridge point of the measured
    # peaks (the dense bf16 rate sustained inside a long step, over the copy bandwidth)
    ridge = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    for name, (n, tot) in sorted(stats.items(), key=lambda kv: -kv[1][1]):
        kind, amount = kernel_work(wl, name, gated, f16_rows)
        avg_s = tot / n * 1e-3
        rate = amount / avg_s if avg_s > 0 else 0.0
        kernels[name] = {"launches": n, "avg_us": round(1e3 * tot / n, 2), "share": round(tot / total_kernel_ms, 4),
                         ("tflops" if kind == "flop" else "gbs"): round(rate / (1e12 if kind == "flop" else 1e9), 1)}
        if kind == "flop":
            nbytes = gemm_bytes(wl, name, experts_used, gated)
            kernels[name]["gbs"] = round(nbytes / avg_s / 1e9, 1) if avg_s > 0 else 0.0
            kernels[name]["flop_per_byte"] = round(amount / nbytes, 1)
    dom = max(stats.items(), key=lambda kv: kv[1][1])[0]
    kind, amount = kernel_work(wl, dom, gated, f16_rows)
    dom_avg_s = stats[dom][1] / stats[dom][0] * 1e-3
    if kind == "flop" and amount / gemm_bytes(wl, dom, experts_used, gated) >= ridge:
        achieved = amount / dom_avg_s / 1e12
        peak = peaks["bf16_tflops_sustained"]
        roofline = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                    "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None,
                    "algorithmic_per_launch": amount,
                    "peak_kind": f"bf16 sustained ({peaks['source']}): timed inside a long step"}
    elif kind == "flop":
        nbytes = gemm_bytes(wl, dom, experts_used, gated)
        achieved = nbytes / dom_avg_s / 1e9
        roofline = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": None,
                    "algorithmic_per_launch": nbytes, "flop_per_launch": amount,
                    "flop_per_byte": round(amount / nbytes, 1), "ridge_flop_per_byte": round(ridge, 1),
                    "peak_kind": f"hbm copy ({peaks['source']})"}
    else:
        achieved = amount / dom_avg_s / 1e9
        roofline = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": None,
                    "algorithmic_per_launch": amount, "peak_kind": f"hbm copy ({peaks['source']})"}
    traffic = load_traffic(wl.name, dom)
    if traffic is not None:
        roofline["traffic"] = traffic

    inf_gemms = gemm_rates(wl, inf_records, peaks, gated)
    inference = {"ms_per_step": round(inf_ms, 4), "tflops": round(whole_job_rate(world, fl["fwd"], inf_ms) / 1e12, 2),
                 "tokens_per_s": round(whole_job_rate(world, T, inf_ms), 1),
                 "saved_state": "none: the forward keeps no derivative factors for a backward",
                 "gemms": inf_gemms}

    # ---------------- end to end: host buffers, copies inside the timed loop
    # Every step uploads its inputs (logits, x, dY) from pinned host memory and downloads its
    # results (Y, dX, d_logits).  As in a training loop, a copy stream moves step i+1's inputs
    # and step i-1's results while step i computes (inputs and results are double-buffered);
    # the timed region spans the first upload to the last download.
    e2e = None
    if not args.no_e2e:
        h_logits = torch.from_numpy(inp["logits"]).pin_memory()
        h_x = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
        h_dy = torch.from_numpy(inp["dy"].view(np.int16)).view(torch.bfloat16).pin_memory()
        d_in = [(torch.empty_like(logits), torch.empty_like(x), torch.empty_like(dy)) for _ in range(2)]
        # uploads per step: (logits,) x, dY -- with --router the logits buffer is written on the device
        up = (lambda b_: list(zip(d_in[b_], (h_logits, h_x, h_dy)))[1 if args.router else 0:])
        d_out = [(e(T, H), e(T, H), e(T, E, dt=f32)) for _ in range(2)]
        h_out = [(torch.empty((T, H), dtype=bf).pin_memory(), torch.empty((T, H), dtype=bf).pin_memory(),
                  torch.empty((T, E), dtype=f32).pin_memory()) for _ in range(2)]
        copy_s = torch.cuda.Stream(device=dev)
        ev = lambda: torch.cuda.Event(enable_timing=False)

        def run_e2e(nsteps):
            cur = torch.cuda.current_stream()
            uploaded = [ev(), ev()]
            computed = [ev(), ev()]
            downloaded = [ev(), ev()]
            start = ev()
            start.record(cur)
            copy_s.wait_event(start)
            with torch.cuda.stream(copy_s):
                for b_ in range(min(2, nsteps)):
                    for dst, src in up(b_):
                        dst.copy_(src, non_blocking=True)
                    uploaded[b_].record(copy_s)
            for i in range(nsteps):
                b_ = i % 2
                cur.wait_event(uploaded[b_])
                if i >= 2:
                    cur.wait_event(downloaded[b_])  # result buffers of step i-2 are on the host
                lg, xx, dyy = d_in[b_]
                Yb, dxb, dlb = d_out[b_]
                forward(lg, xx, y_out=Yb)
                backward(dyy, xx, dx_out=dxb, dl_out=dlb)
                computed[b_].record(cur)
                copy_s.wait_event(computed[b_])
                with torch.cuda.stream(copy_s):
                    for dst, src in zip(h_out[b_], (Yb, dxb, dlb)):
                        dst.copy_(src, non_blocking=True)
                    downloaded[b_].record(copy_s)
                    if i + 2 < nsteps:  # next inputs into this buffer once step i has consumed it
                        for dst, src in up(b_):
                            dst.copy_(src, non_blocking=True)
                        uploaded[b_].record(copy_s)
            cur.wait_stream(copy_s)

        run_e2e(3)
        torch.cuda.synchronize()
        ne = max(3, args.steps // 2)
        g2 = None
        if graph is not None:
            try:
                g2 = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g2):
                    run_e2e(ne)
                g2.replay()
                torch.cuda.synchronize()
            except Exception:
                g2 = None
                torch.cuda.synchronize()
        barrier()
        ev4, ev5 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev4.record(stream)
        if g2 is not None:
            g2.replay()
        else:
            run_e2e(ne)
        ev5.record(stream)
        torch.cuda.synchronize()
        barrier()
        e2e_ms = max_over_ranks(ev4.elapsed_time(ev5))
        h2d = (0 if args.router else T * E * 4) + 2 * T * H * 2
        d2h = 2 * T * H * 2 + T * E * 4
        e2e = {"value": round(whole_job_rate(world, ne * fl["total"], e2e_ms) / 1e12, 2), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / ne, 4),
               "weights": "resident on the device; dW stays on the device",
               "copies": "double-buffered on a copy stream, overlapped with the neighbouring steps' compute",
               "graph": g2 is not None}

    # ---------------- the training shape's forward GEMMs (tensor-bound there), own buffers
    tsf = None
    if not args.no_train_shape:
        tsf = train_shape_forward(args, dev, local_rank, peaks, max_over_ranks, world)

    # ---------------- CPU oracle baseline (rank 0, one GPU only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        ids_h, w_h = oracle.route_topk(inp["logits"], k)
        n_tok, experts = size_oracle_sample(wl, inp, ids_h, w_h, args.cpu_seconds, (args.act, args.act_clamp),
                                            args.router)
        t0 = time.perf_counter()
        f = oracle_sample(wl, inp, ids_h, w_h, n_tok, experts, (args.act, args.act_clamp), args.router)
        dt = time.perf_counter() - t0
        cpu = {"value": round(f / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.default_threads(),
               "kind": "oracle",
               "sample": f"forward + dX + d_logits{' + router projection and its backward' if args.router else ''} "
                         f"of tokens 0..{n_tok - 1} of {T}, dW of {len(experts)} experts ({dt:.1f} s wall)"}

    launches = sum(launch_counts)  # kernels of the timed steps (a split GEMM's interval holds two)
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(wl.as_dict(), **{"pass": "forward+backward", "parallelism": f"replicas x{world}",
                                           "expert_inputs": args.inputs, "activation": args.act,
                                           "dw_operands": (f"fp16 (scaled by powers of two) for the {f16_rows} routed "
                                                           "rows of experts with 384+ rows; bf16 hi + lo for the rest"
                                                           if f16_rows else "bf16 hi + lo"),
                                           "router": "x Wr^T (+ bias) and its backward on the GPU" if args.router
                                           else "logits are the layer's input",
                                           "l2": f"inputs larger than L2: {L.weight_bytes / 1e9:.2f} GB "
                                                 f"of weights + activations streamed per step (L2 129 MB)"}),
            "tokens_per_s": round(tokens_per_s, 1),
            "fwd_ms": round(fwd_ms, 4), "bwd_ms": round(ms_per_step - fwd_ms, 4),
            "fwd_tflops": round(whole_job_rate(world, fl["fwd"], fwd_ms) / 1e12, 2),
            "bwd_tflops": round(whole_job_rate(world, fl["bwd"], ms_per_step - fwd_ms) / 1e12, 2),
            "pct_of_bf16_peak": round(100 * value / world / peaks["bf16_tflops"], 2),
            "inference_forward": inference, "sustained": sustained, "train_shape_forward": tsf,
            "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches, "clocks": clock_info, "launch": graph_note,
            "traced_ms_per_step": None if trace_ms is None else round(trace_ms, 4),
        }
        print(json.dumps(line), flush=True)


def kernel_source_hash() -> str:
    """sha256 over the GEMM kernel's sources (the kernel file and its inline-PTX header)."""
    import hashlib

    h = hashlib.sha256()
    for name in ("grouped_gemm.cu", "ptx.cuh"):
        with open(os.path.join(ROOT, "mixture_experts_routed_router_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def load_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of `kernel` from a committed ncu capture, if one matches.

    None when there is no capture for this workload and kernel, or when the GEMM source
    has changed since the counters were taken (the capture records its hash).
    """
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            entry = json.load(f)[workload][kernel]
        if kernel_source_hash() != entry.get("kernel_source_sha256"):
            return None
        return entry["dram_bytes_per_launch"]
    except (OSError, KeyError, ValueError, TypeError):
        return None


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
