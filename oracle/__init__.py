"""CPU oracle of the routed MoE layer (forward and backward).

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke``
and by the CPU-baseline leg of ``bench.py``; never by the product path.
It shares no code with the CUDA library.  The arithmetic lives in
``moe_oracle.cpp`` (plain loops, float accumulation from bf16 inputs,
compiled with ``-ffp-contract=off``); this module only marshals numpy
arrays.  bf16 tensors are numpy ``uint16`` bit patterns.

Every function is pinned by tests that do not call it to get their expected
values (brute force, fp64 dense evaluation, autograd, finite differences,
closed forms, degenerate cases): see ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def compile_source(src: str, out: str) -> str:
    """g++ of one oracle source into a shared library (plain C++17, no fused multiply-add)."""
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile moe_oracle.cpp into liboracle.so beside it (skipped when up to date)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def open_library(path: str):
    """Load an oracle build (the default one, or a test's planted-mistake copy)."""
    lib = ctypes.CDLL(path)
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.oracle_route_topk.argtypes = [P, I, I, I, P, P]
    lib.oracle_dispatch.argtypes = [P, P, P, I, I, I, I, P, P, P, P, P, P]
    F = ctypes.c_float
    lib.oracle_grouped_swiglu_rows.argtypes = [P, P, P, P, P, I, I, I, I, P, I, P, P, P, I, F, I]
    lib.oracle_combine.argtypes = [P, P, I, I, I, P, I, P]
    lib.oracle_forward_tokens.argtypes = [P, P, P, P, P, I, I, I, I, I, P, I, P, I, F, I]
    lib.oracle_backward_tokens.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, I, P, P, I, F, I]
    lib.oracle_backward_dw.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, I, P, P, I, F, I]
    lib.oracle_router_logits.argtypes = [P, P, P, I, I, I, P, I]
    lib.oracle_router_backward.argtypes = [P, P, P, P, I, I, I, P, I, P, P, I, P, P, I]
    for f in (lib.oracle_route_topk, lib.oracle_dispatch, lib.oracle_grouped_swiglu_rows,
              lib.oracle_combine, lib.oracle_forward_tokens, lib.oracle_backward_tokens,
              lib.oracle_backward_dw, lib.oracle_router_logits, lib.oracle_router_backward):
        f.restype = ctypes.c_int
    return lib


_override = threading.local()


def _load():
    lib = getattr(_override, "lib", None)
    if lib is not None:
        return lib
    global _lib
    with _lock:
        if _lib is None:
            _lib = open_library(build())
    return _lib


class using:
    """Context manager: run the module functions on another oracle build (tests only)."""

    def __init__(self, lib):
        self.lib = lib

    def __enter__(self):
        self.prev = getattr(_override, "lib", None)
        _override.lib = self.lib
        return self

    def __exit__(self, *exc):
        _override.lib = self.prev
        return False


# Activations of the expert MLP (moe_oracle.cpp, act_forward); `clamp` is the bound of the
# bounded SwiGLU and the limit of SwiGLU-OAI, unused otherwise.  All but relu2 are gated and take
# wgu [E, 2I, H] (gate rows, then up rows); relu2 takes the up weight [E, I, H] in its place.
ACTIVATIONS = {"swiglu": 0, "swiglu_bounded": 1, "swiglu_oai": 2, "geglu": 3, "reglu": 4, "relu2": 5}


def _act(act: str) -> int:
    if act not in ACTIVATIONS:
        raise ValueError(f"unknown activation {act!r}")
    return ACTIVATIONS[act]


def _inter(wgu, act: str) -> int:
    """I from the first weight's rows: 2I for the gated activations, I for relu2."""
    rows = wgu.shape[1]
    return rows if act == "relu2" else rows // 2


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _check(rc: int, name: str):
    if rc != 0:
        raise ValueError(f"oracle {name} rejected its arguments (status {rc})")


def route_topk(logits: np.ndarray, k: int):
    """Returns (ids int32 [T,k], w float32 [T,k])."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    _check(_load().oracle_route_topk(logits.ctypes.data, T, E, k, ids.ctypes.data, w.ctypes.data), "route_topk")
    return ids, w


def dispatch(ids: np.ndarray, w: np.ndarray | None, x: np.ndarray | None, E: int):
    """Returns dict(counts, m_indptr, row_to_slot, slot_to_row, w_perm, x_perm)."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    R = T * k
    H = 0 if x is None else x.shape[1]
    x = None if x is None else _c(x, np.uint16)
    w = None if w is None else _c(w, np.float32)
    out = dict(counts=np.empty(E, np.int32), m_indptr=np.empty(E + 1, np.int32),
               row_to_slot=np.empty(R, np.int32), slot_to_row=np.empty(R, np.int32),
               w_perm=None if w is None else np.empty(R, np.float32),
               x_perm=None if x is None else np.empty((R, H), np.uint16))
    rc = _load().oracle_dispatch(ids.ctypes.data, _ptr(w), _ptr(x), T, H, E, k,
                                 out["counts"].ctypes.data, out["m_indptr"].ctypes.data,
                                 out["row_to_slot"].ctypes.data, out["slot_to_row"].ctypes.data,
                                 _ptr(out["w_perm"]), _ptr(out["x_perm"]))
    _check(rc, "dispatch")
    return out


def grouped_swiglu_rows(x_perm, m_indptr, wgu, wd, w_perm, rows, threads=None, act="swiglu", clamp=0.0):
    """Expert MLP on chosen expert-major rows: (h bf16 [n,I], gu f32 [n,2I] = [g | u], y bf16 [n,H]).

    relu2: gu is [n, I] (its one projection)."""
    x_perm = _c(x_perm, np.uint16)
    wgu = _c(wgu, np.uint16)
    wd = _c(wd, np.uint16)
    m_indptr = _c(m_indptr, np.int32)
    w_perm = _c(w_perm, np.float32)
    rows = _c(rows, np.int32)
    R, H = x_perm.shape
    E, nin, _ = wgu.shape
    I = _inter(wgu, act)
    n = rows.size
    h = np.empty((n, I), np.uint16)
    gu = np.empty((n, nin), np.float32)
    y = np.empty((n, H), np.uint16)
    rc = _load().oracle_grouped_swiglu_rows(x_perm.ctypes.data, m_indptr.ctypes.data, wgu.ctypes.data,
                                            wd.ctypes.data, w_perm.ctypes.data, R, H, I, E, rows.ctypes.data,
                                            n, h.ctypes.data, gu.ctypes.data, y.ctypes.data, _act(act),
                                            float(clamp), threads or default_threads())
    _check(rc, "grouped_swiglu_rows")
    return h, gu, y


def combine(y_perm, slot_to_row, T, k, toks=None):
    y_perm = _c(y_perm, np.uint16)
    slot_to_row = _c(slot_to_row, np.int32)
    H = y_perm.shape[1]
    toks = np.arange(T, dtype=np.int32) if toks is None else _c(toks, np.int32)
    out = np.empty((toks.size, H), np.uint16)
    _check(_load().oracle_combine(y_perm.ctypes.data, slot_to_row.ctypes.data, T, H, k, toks.ctypes.data,
                                  toks.size, out.ctypes.data), "combine")
    return out


def forward_tokens(x, wgu, wd, ids, w, toks=None, threads=None, act="swiglu", clamp=0.0):
    """Whole-layer output Y (bf16 [n,H]) for the listed tokens."""
    x, wgu, wd = _c(x, np.uint16), _c(wgu, np.uint16), _c(wd, np.uint16)
    ids, w = _c(ids, np.int32), _c(w, np.float32)
    T, H = x.shape
    E = wgu.shape[0]
    k = ids.shape[1]
    toks = np.arange(T, dtype=np.int32) if toks is None else _c(toks, np.int32)
    out = np.empty((toks.size, H), np.uint16)
    rc = _load().oracle_forward_tokens(x.ctypes.data, wgu.ctypes.data, wd.ctypes.data, ids.ctypes.data,
                                       w.ctypes.data, T, H, _inter(wgu, act), E, k, toks.ctypes.data, toks.size,
                                       out.ctypes.data, _act(act), float(clamp), threads or default_threads())
    _check(rc, "forward_tokens")
    return out


def backward_tokens(x, dy, wgu, wd, ids, w, toks=None, threads=None, act="swiglu", clamp=0.0):
    """(dX bf16 [n,H], d_logits float32 [n,E]) for the listed tokens."""
    x, dy = _c(x, np.uint16), _c(dy, np.uint16)
    wgu, wd = _c(wgu, np.uint16), _c(wd, np.uint16)
    ids, w = _c(ids, np.int32), _c(w, np.float32)
    T, H = x.shape
    E = wgu.shape[0]
    k = ids.shape[1]
    toks = np.arange(T, dtype=np.int32) if toks is None else _c(toks, np.int32)
    dx = np.empty((toks.size, H), np.uint16)
    dl = np.empty((toks.size, E), np.float32)
    rc = _load().oracle_backward_tokens(x.ctypes.data, dy.ctypes.data, wgu.ctypes.data, wd.ctypes.data,
                                        ids.ctypes.data, w.ctypes.data, T, H, _inter(wgu, act), E, k,
                                        toks.ctypes.data, toks.size, dx.ctypes.data, dl.ctypes.data,
                                        _act(act), float(clamp), threads or default_threads())
    _check(rc, "backward_tokens")
    return dx, dl


def backward_dw(x, dy, wgu, wd, ids, w, experts=None, threads=None, act="swiglu", clamp=0.0):
    """(dW_gu bf16 [n,2I,H] (relu2: [n,I,H]), dW_d bf16 [n,H,I]) for the listed experts."""
    x, dy = _c(x, np.uint16), _c(dy, np.uint16)
    wgu, wd = _c(wgu, np.uint16), _c(wd, np.uint16)
    ids, w = _c(ids, np.int32), _c(w, np.float32)
    T, H = x.shape
    E, nin, _ = wgu.shape
    I = _inter(wgu, act)
    k = ids.shape[1]
    experts = np.arange(E, dtype=np.int32) if experts is None else _c(experts, np.int32)
    dwgu = np.empty((experts.size, nin, H), np.uint16)
    dwd = np.empty((experts.size, H, I), np.uint16)
    rc = _load().oracle_backward_dw(x.ctypes.data, dy.ctypes.data, wgu.ctypes.data, wd.ctypes.data,
                                    ids.ctypes.data, w.ctypes.data, T, H, I, E, k, experts.ctypes.data,
                                    experts.size, dwgu.ctypes.data, dwd.ctypes.data, _act(act), float(clamp),
                                    threads or default_threads())
    _check(rc, "backward_dw")
    return dwgu, dwd


def router_logits(x, wr, bias=None, threads=None):
    """Router projection logits = x Wr^T + bias (float32 [T, E]); bias float32 [E] or None."""
    x, wr = _c(x, np.uint16), _c(wr, np.uint16)
    T, H = x.shape
    E = wr.shape[0]
    if wr.shape != (E, H):
        raise ValueError("wr must be [E, H]")
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((T, E), np.float32)
    rc = _load().oracle_router_logits(x.ctypes.data, wr.ctypes.data, _ptr(b), T, H, E, out.ctypes.data,
                                      threads or default_threads())
    _check(rc, "router_logits")
    return out


def router_backward(d_logits, x, wr, dx_in=None, toks=None, experts=None, threads=None):
    """(dX bf16 [n, H] = bf16(dx_in + d_logits Wr) for the listed tokens, dWr bf16 [m, H] and
    dbias float32 [m] for the listed experts); d_logits float32 [T, E] is used densely."""
    dl = _c(d_logits, np.float32)
    x, wr = _c(x, np.uint16), _c(wr, np.uint16)
    T, H = x.shape
    E = wr.shape[0]
    if dl.shape != (T, E) or wr.shape != (E, H):
        raise ValueError("d_logits must be [T, E] and wr [E, H]")
    base = None if dx_in is None else _c(dx_in, np.uint16)
    if base is not None and base.shape != (T, H):
        raise ValueError("dx_in must be [T, H]")
    toks = np.arange(T, dtype=np.int32) if toks is None else _c(toks, np.int32)
    experts = np.arange(E, dtype=np.int32) if experts is None else _c(experts, np.int32)
    dx = np.empty((toks.size, H), np.uint16)
    dwr = np.empty((experts.size, H), np.uint16)
    db = np.empty(experts.size, np.float32)
    rc = _load().oracle_router_backward(dl.ctypes.data, x.ctypes.data, wr.ctypes.data, _ptr(base), T, H, E,
                                        toks.ctypes.data, toks.size, dx.ctypes.data, experts.ctypes.data,
                                        experts.size, dwr.ctypes.data, db.ctypes.data,
                                        threads or default_threads())
    _check(rc, "router_backward")
    return dx, dwr, db
