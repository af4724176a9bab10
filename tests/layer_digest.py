"""Runs one routed MoE layer step (forward and backward) on cuda:0 and prints the SHA-256 of
every output, as launched one call at a time and as replayed from a captured CUDA graph (or, with
"capture_first", only the latter, captured before any other call).

Used by tests/test_gpu_pdl.py as a child process: the library reads its launch mode
(LIGER_MOE_PDL=1: programmatic dependent launch; =0: plain stream order; unset: programmatic
launch for the calls below 4096 routed rows) once per process, so each mode gets its own process.  Every kernel sums in a fixed order, so the digests must not depend on
the launch mode or on graph replay.
"""
from __future__ import annotations

import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import mixture_experts_routed_router_gb300 as moe  # noqa: E402
import synthetic  # noqa: E402


def _dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def _digest(t: torch.Tensor) -> str:
    t = t.detach().contiguous()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return hashlib.sha256(t.cpu().numpy().tobytes()).hexdigest()


def main() -> None:
    wl = synthetic.workload(sys.argv[1])
    # "capture_first": the process's first library calls are made inside the graph capture (the
    # backward then finds no side stream and runs in order on the captured stream)
    capture_first = len(sys.argv) > 2 and sys.argv[2] == "capture_first"
    inp = synthetic.make_inputs(wl)
    logits, x, dy = _dev(inp["logits"]), _dev(inp["x"]), _dev(inp["dy"])
    wgu, wd = _dev(inp["wgu"]), _dev(inp["wd"])

    def step() -> dict:
        ids, w = moe.route_topk(logits, wl.k)
        d = moe.dispatch(ids, w, x, wl.E)
        h, gu, y_perm = moe.grouped_swiglu_fwd(d["x_perm"], d["m_indptr"], wgu, wd, d["w_perm"])
        Y = moe.combine(y_perm, d["slot_to_row"], wl.T, wl.k)
        dx, dwgu, dwd, dl = moe.bwd_dx_dw(dy, d["x_perm"], h, gu, ids, w, d["m_indptr"], d["row_to_slot"],
                                          d["slot_to_row"], d["w_perm"], wgu, wd)
        return dict(ids=ids, w=w, m_indptr=d["m_indptr"], row_to_slot=d["row_to_slot"], x_perm=d["x_perm"], h=h,
                    gu=gu, Y=Y, dx=dx, dw_gate_up=dwgu, dw_down=dwd, d_logits=dl)

    out = {}
    if not capture_first:
        eager = step()
        torch.cuda.synchronize()
        out["eager"] = {k: _digest(v) for k, v in eager.items()}
        step()  # warm the allocator before capture
        torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        captured = step()
    graph.replay()
    torch.cuda.synchronize()
    out["graph"] = {k: _digest(v) for k, v in captured.items()}
    out["device_error"] = moe.device_error()
    print(json.dumps(out))


if __name__ == "__main__":
    main()
