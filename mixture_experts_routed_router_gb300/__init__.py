"""Routed Mixture-of-Experts layer (forward + backward) on one GB300: Python binding.

Every computation runs in ``libliger_moe.so`` (hand-written CUDA for sm_103a,
see ``include/liger_moe.h``).  This module only checks tensor dtypes, shapes
and devices, allocates outputs with PyTorch when the caller does not pass
them, and calls the C entry points of the same names on the current CUDA
stream.  There is no fallback: without the library, or without an sm_103
device, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

__all__ = ["route_topk", "dispatch", "grouped_swiglu_fwd", "grouped_swiglu_fwd_gather", "grouped_glu_fwd",
           "combine", "bwd_dx_dw", "bwd_dx_dw_gather", "bwd_dx_dw_glu", "router_logits", "router_bwd", "ACTIVATIONS",
           "device_error",
           "selftest_wait_timeout", "workspace_bytes", "set_dw_fp16", "trace_enable", "trace_records", "LigerMoEError", "library_path", "load_library"]

_lock = threading.Lock()
_lib = None

OK = 0
STATUS = {0: "OK", -1: "INVALID_ARG", -2: "MISALIGNED", -3: "CAPACITY", -4: "UNSUPPORTED_DEVICE", -5: "LAUNCH",
          -6: "DEVICE"}
DEVERR = {0x1: "BAD_EXPERT_ID", 0x2: "BAD_ROW", 0x4: "BAD_INDPTR", 0x8: "WAIT_TIMEOUT"}
# enum liger_moe_activation: activations of the expert MLP (relu2: two-weight, non-gated experts)
ACTIVATIONS = {"swiglu": 0, "swiglu_bounded": 1, "swiglu_oai": 2, "geglu": 3, "reglu": 4, "relu2": 5}


class LigerMoEError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}{(' (' + detail + ')') if detail else ''}")


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = True):
    """Loads libliger_moe.so (building it with nvcc first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build() if build_if_missing else _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libliger_moe.so not found at {path}")
        lib = ctypes.CDLL(path)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)
        lib.liger_moe_route_topk.argtypes = [P, I, I, I, P, P, P]
        lib.liger_moe_dispatch.argtypes = [P, P, P, I, I, I, I, P, P, P, P, P, P, P, S, P]
        lib.liger_moe_grouped_swiglu_fwd.argtypes = [P, P, P, P, P, I, I, I, I, P, P, P, P, S, P]
        lib.liger_moe_combine.argtypes = [P, P, I, I, I, P, P]
        lib.liger_moe_bwd_dx_dw.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, P, P, P, P, P, S, P]
        lib.liger_moe_grouped_swiglu_fwd_gather.argtypes = [P, P, I, I, P, P, P, P, I, I, I, P, P, P, P, S, P]
        lib.liger_moe_bwd_dx_dw_gather.argtypes = lib.liger_moe_bwd_dx_dw.argtypes
        F = ctypes.c_float
        lib.liger_moe_grouped_glu_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, F, P, P, P, P, S, P]
        lib.liger_moe_bwd_dx_dw_glu.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P, P, P, P,
                                                P, S, P]
        lib.liger_moe_router_logits.argtypes = [P, P, P, I, I, I, P, P]
        lib.liger_moe_router_bwd.argtypes = [P, P, P, P, P, P, I, I, I, I, P, P, P, P]
        lib.liger_moe_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_int)]
        lib.liger_moe_selftest_wait_timeout.argtypes = [I, P]
        lib.liger_moe_trace_enable.argtypes = [I]
        lib.liger_moe_set_dw_fp16.argtypes = [I]
        lib.liger_moe_trace_get.argtypes = [I, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float)]
        lib.liger_moe_trace_launches.argtypes = [I, ctypes.POINTER(ctypes.c_int)]
        lib.liger_moe_last_cuda_error.restype = ctypes.c_char_p
        lib.liger_moe_status_string.restype = ctypes.c_char_p
        lib.liger_moe_status_string.argtypes = [I]
        for f in (lib.liger_moe_route_topk, lib.liger_moe_dispatch, lib.liger_moe_grouped_swiglu_fwd,
                  lib.liger_moe_grouped_swiglu_fwd_gather, lib.liger_moe_combine, lib.liger_moe_bwd_dx_dw,
                  lib.liger_moe_bwd_dx_dw_gather, lib.liger_moe_grouped_glu_fwd, lib.liger_moe_bwd_dx_dw_glu,
                  lib.liger_moe_router_logits, lib.liger_moe_router_bwd, lib.liger_moe_device_error,
                  lib.liger_moe_selftest_wait_timeout,
                  lib.liger_moe_abi_version, lib.liger_moe_trace_enable, lib.liger_moe_trace_count,
                  lib.liger_moe_trace_get, lib.liger_moe_trace_launches, lib.liger_moe_set_dw_fp16):
            f.restype = ctypes.c_int
        _lib = lib
        return lib


def _check(fn: str, rc: int):
    if rc != OK:
        lib = load_library()
        raise LigerMoEError(fn, rc, lib.liger_moe_last_cuda_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def _out(t, name, dtype, shape, device):
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    return _need(t, name, dtype, shape)


def _workspace(ws, nbytes, device):
    if ws is None:
        return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    _need(ws, "workspace", torch.uint8)
    if ws.numel() < nbytes:
        raise ValueError(f"workspace has {ws.numel()} bytes, {nbytes} needed")
    return ws


def router_logits(x, w_router, bias=None, *, out=None, stream=None):
    """Router projection logits = x w_router^T (+ bias): float32 [T, E] from x bf16 [T, H],
    w_router bf16 [E, H] and bias float32 [E] or None."""
    lib = load_library()
    _need(x, "x", torch.bfloat16)
    T, H = x.shape
    _need(w_router, "w_router", torch.bfloat16)
    E = w_router.shape[0]
    _need(w_router, "w_router", torch.bfloat16, (E, H))
    if bias is not None:
        _need(bias, "bias", torch.float32, (E,))
    out = _out(out, "logits", torch.float32, (T, E), x.device)
    _check("liger_moe_router_logits", lib.liger_moe_router_logits(_ptr(x), _ptr(w_router), _ptr(bias), T, H, E,
                                                                  _ptr(out), _stream(stream)))
    return out


def router_bwd(d_logits, topk_ids, m_indptr, row_to_slot, x, w_router, dx, *, dw_router=None, d_bias=None,
               want_bias=True, stream=None):
    """Backward of the router projection for the layer's d_logits (zero off the top-k).

    Adds the router's input gradient to dx (bf16 [T, H], updated in place) and returns
    (dw_router bf16 [E, H], d_bias float32 [E] or None when want_bias is False)."""
    lib = load_library()
    _need(d_logits, "d_logits", torch.float32)
    T, E = d_logits.shape
    _need(topk_ids, "topk_ids", torch.int32)
    k = topk_ids.shape[1]
    _need(x, "x", torch.bfloat16)
    H = x.shape[1]
    for t, n, dt, sh in ((topk_ids, "topk_ids", torch.int32, (T, k)), (m_indptr, "m_indptr", torch.int32, (E + 1,)),
                         (row_to_slot, "row_to_slot", torch.int32, (T * k,)), (x, "x", torch.bfloat16, (T, H)),
                         (w_router, "w_router", torch.bfloat16, (E, H)), (dx, "dx", torch.bfloat16, (T, H))):
        _need(t, n, dt, sh)
    dw_router = _out(dw_router, "dw_router", torch.bfloat16, (E, H), x.device)
    d_bias = _out(d_bias, "d_bias", torch.float32, (E,), x.device) if want_bias else None
    _check("liger_moe_router_bwd", lib.liger_moe_router_bwd(
        _ptr(d_logits), _ptr(topk_ids), _ptr(m_indptr), _ptr(row_to_slot), _ptr(x), _ptr(w_router), T, H, E, k,
        _ptr(dx), _ptr(dw_router), _ptr(d_bias), _stream(stream)))
    return dw_router, d_bias


def route_topk(logits, k, *, topk_ids=None, topk_w=None, stream=None):
    """(topk_ids int32 [T,k], topk_w float32 [T,k]) from logits float32 [T,E]."""
    lib = load_library()
    _need(logits, "logits", torch.float32)
    T, E = logits.shape
    topk_ids = _out(topk_ids, "topk_ids", torch.int32, (T, k), logits.device)
    topk_w = _out(topk_w, "topk_w", torch.float32, (T, k), logits.device)
    _check("liger_moe_route_topk", lib.liger_moe_route_topk(_ptr(logits), T, E, k, _ptr(topk_ids), _ptr(topk_w),
                                                            _stream(stream)))
    return topk_ids, topk_w


def workspace_bytes(fn: str, **kw) -> int:
    """Workspace size an entry point needs (query call: nothing is launched)."""
    lib = load_library()
    n = ctypes.c_size_t(0)
    d = ctypes.c_void_p(256)  # stand-in pointers: a query validates arguments but never dereferences them
    if fn == "dispatch":
        T, E, k = kw["T"], kw["E"], kw["k"]
        rc = lib.liger_moe_dispatch(d, None, None, T, 0, E, k, d, d, d, d, None, None, None, ctypes.byref(n), None)
    elif fn == "grouped_swiglu_fwd":
        R, H, I, E = kw["R"], kw["H"], kw["I"], kw["E"]
        p = None if R == 0 else ctypes.c_void_p(256)
        rc = lib.liger_moe_grouped_swiglu_fwd(p, ctypes.c_void_p(256), p, p, p, R, H, I, E, p, None, p, None,
                                              ctypes.byref(n), None)
    elif fn == "bwd_dx_dw":
        T, H, I, E, k = kw["T"], kw["H"], kw["I"], kw["E"], kw["k"]
        p = ctypes.c_void_p(256)
        q = None if T * k == 0 else p
        gu = p if kw.get("saved_gu", True) else None
        f = lib.liger_moe_bwd_dx_dw_gather if kw.get("gather", False) else lib.liger_moe_bwd_dx_dw
        rc = f(q, q, q, gu, q, q, p, q, q, q, p, p, T, H, I, E, k, q, p, p, q, None, ctypes.byref(n), None)
    else:
        raise ValueError(fn)
    _check(f"workspace query ({fn})", rc)
    return n.value


def dispatch(topk_ids, topk_w, x, num_experts, *, out=None, workspace=None, stream=None):
    """Deterministic expert-major dispatch.

    Returns dict(counts, m_indptr, row_to_slot, slot_to_row, w_perm, x_perm); w_perm / x_perm
    are None when topk_w / x is None.
    """
    lib = load_library()
    _need(topk_ids, "topk_ids", torch.int32)
    T, k = topk_ids.shape
    R, E, dev = T * k, num_experts, topk_ids.device
    H = 0 if x is None else x.shape[1]
    if topk_w is not None:
        _need(topk_w, "topk_w", torch.float32, (T, k))
    if x is not None:
        _need(x, "x", torch.bfloat16, (T, H))
    out = dict(out or {})
    o = dict(counts=_out(out.get("counts"), "counts", torch.int32, (E,), dev),
             m_indptr=_out(out.get("m_indptr"), "m_indptr", torch.int32, (E + 1,), dev),
             row_to_slot=_out(out.get("row_to_slot"), "row_to_slot", torch.int32, (R,), dev),
             slot_to_row=_out(out.get("slot_to_row"), "slot_to_row", torch.int32, (R,), dev),
             w_perm=None if topk_w is None else _out(out.get("w_perm"), "w_perm", torch.float32, (R,), dev),
             x_perm=None if x is None else _out(out.get("x_perm"), "x_perm", torch.bfloat16, (R, H), dev))
    ws = _workspace(workspace, workspace_bytes("dispatch", T=T, H=H, E=E, k=k), dev)
    n = ctypes.c_size_t(ws.numel())
    _check("liger_moe_dispatch", lib.liger_moe_dispatch(
        _ptr(topk_ids), _ptr(topk_w), _ptr(x), T, H, E, k, _ptr(o["counts"]), _ptr(o["m_indptr"]),
        _ptr(o["row_to_slot"]), _ptr(o["slot_to_row"]), _ptr(o["w_perm"]), _ptr(o["x_perm"]), _ptr(ws),
        ctypes.byref(n), _stream(stream)))
    return o


def _fwd_args(R, H, w_gate_up, w_down, m_indptr, w_perm, save_gu, out, workspace, dev, gated=True):
    _need(w_gate_up, "w_gate_up", torch.bfloat16)
    E, nin, _ = w_gate_up.shape  # gated: [E, 2I, H]; relu2: the up weight [E, I, H]
    I = nin // 2 if gated else nin
    _need(w_gate_up, "w_gate_up", torch.bfloat16, (E, 2 * I if gated else I, H))
    _need(w_down, "w_down", torch.bfloat16, (E, H, I))
    _need(m_indptr, "m_indptr", torch.int32, (E + 1,))
    _need(w_perm, "w_perm", torch.float32, (R,))
    out = dict(out or {})
    h = _out(out.get("h_perm"), "h_perm", torch.bfloat16, (R, I), dev)
    gu = _out(out.get("gu_perm"), "gu_perm", torch.float32, (R, 2 * I if gated else I), dev) if save_gu else None
    y = _out(out.get("y_perm"), "y_perm", torch.bfloat16, (R, H), dev)
    ws = _workspace(workspace, workspace_bytes("grouped_swiglu_fwd", R=R, H=H, I=I, E=E), dev)
    return E, I, h, gu, y, ws


def grouped_swiglu_fwd(x_perm, m_indptr, w_gate_up, w_down, w_perm, *, save_gu=True, out=None, workspace=None,
                       stream=None):
    """Grouped SwiGLU expert MLP: returns (h_perm [R,I] bf16, gu_perm [R,2I] fp32 or None, y_perm [R,H] bf16)."""
    lib = load_library()
    _need(x_perm, "x_perm", torch.bfloat16)
    R, H = x_perm.shape
    E, I, h, gu, y, ws = _fwd_args(R, H, w_gate_up, w_down, m_indptr, w_perm, save_gu, out, workspace, x_perm.device)
    n = ctypes.c_size_t(ws.numel())
    _check("liger_moe_grouped_swiglu_fwd", lib.liger_moe_grouped_swiglu_fwd(
        _ptr(x_perm), _ptr(m_indptr), _ptr(w_gate_up), _ptr(w_down), _ptr(w_perm), R, H, I, E, _ptr(h), _ptr(gu),
        _ptr(y), _ptr(ws), ctypes.byref(n), _stream(stream)))
    return h, gu, y


def _act_id(activation: str) -> int:
    if activation not in ACTIVATIONS:
        raise ValueError(f"unknown activation {activation!r}; one of {sorted(ACTIVATIONS)}")
    return ACTIVATIONS[activation]


def grouped_glu_fwd(x_perm, m_indptr, w_gate_up, w_down, w_perm, activation="swiglu", clamp=0.0, *, save_gu=True,
                    out=None, workspace=None, stream=None):
    """The expert MLP with a chosen activation (ACTIVATIONS); returns (h_perm, gu_perm, y_perm).

    gu_perm holds that activation's derivative factors [dh/dg | dh/du]; clamp is the bound of
    swiglu_bounded and the limit of swiglu_oai.  relu2 (two-weight experts): w_gate_up is the
    up weight [E, I, H] and gu_perm [R, I] holds dh/da.
    """
    lib = load_library()
    _need(x_perm, "x_perm", torch.bfloat16)
    R, H = x_perm.shape
    E, I, h, gu, y, ws = _fwd_args(R, H, w_gate_up, w_down, m_indptr, w_perm, save_gu, out, workspace, x_perm.device,
                                   gated=activation != "relu2")
    n = ctypes.c_size_t(ws.numel())
    _check("liger_moe_grouped_glu_fwd", lib.liger_moe_grouped_glu_fwd(
        _ptr(x_perm), _ptr(m_indptr), _ptr(w_gate_up), _ptr(w_down), _ptr(w_perm), R, H, I, E, _act_id(activation),
        float(clamp), _ptr(h), _ptr(gu), _ptr(y), _ptr(ws), ctypes.byref(n), _stream(stream)))
    return h, gu, y


def grouped_swiglu_fwd_gather(x, row_to_slot, k, m_indptr, w_gate_up, w_down, w_perm, *, save_gu=True, out=None,
                              workspace=None, stream=None):
    """The expert MLP on token-major x [T,H]: row r reads x[row_to_slot[r] // k] (no x_perm).

    Returns (h_perm, gu_perm or None, y_perm) as grouped_swiglu_fwd.
    """
    lib = load_library()
    _need(x, "x", torch.bfloat16)
    T, H = x.shape
    R = T * k
    _need(row_to_slot, "row_to_slot", torch.int32, (R,))
    E, I, h, gu, y, ws = _fwd_args(R, H, w_gate_up, w_down, m_indptr, w_perm, save_gu, out, workspace, x.device)
    n = ctypes.c_size_t(ws.numel())
    _check("liger_moe_grouped_swiglu_fwd_gather", lib.liger_moe_grouped_swiglu_fwd_gather(
        _ptr(x), _ptr(row_to_slot), T, k, _ptr(m_indptr), _ptr(w_gate_up), _ptr(w_down), _ptr(w_perm), H, I, E,
        _ptr(h), _ptr(gu), _ptr(y), _ptr(ws), ctypes.byref(n), _stream(stream)))
    return h, gu, y


def combine(y_perm, slot_to_row, T, k, *, out=None, stream=None):
    """Y [T,H] = bf16(sum_j y_perm[slot_to_row[t*k+j]])."""
    lib = load_library()
    _need(y_perm, "y_perm", torch.bfloat16)
    H = y_perm.shape[1]
    _need(slot_to_row, "slot_to_row", torch.int32, (T * k,))
    y = _out(out, "y", torch.bfloat16, (T, H), y_perm.device)
    _check("liger_moe_combine", lib.liger_moe_combine(_ptr(y_perm), _ptr(slot_to_row), T, H, k, _ptr(y),
                                                      _stream(stream)))
    return y


def _bwd(fn, dy, x_src, x_name, h_perm, gu_perm, topk_ids, topk_w, m_indptr, row_to_slot, slot_to_row, w_perm,
         w_gate_up, w_down, out, workspace, stream, act=None):
    lib = load_library()
    _need(dy, "dy", torch.bfloat16)
    T, H = dy.shape
    _need(topk_ids, "topk_ids", torch.int32)
    k = topk_ids.shape[1]
    E, nin, _ = w_gate_up.shape  # gated: [E, 2I, H]; relu2: the up weight [E, I, H]
    gated = act is None or act[0] != "relu2"
    I = nin // 2 if gated else nin
    nin = 2 * I if gated else I
    R = T * k
    x_shape = (T, H) if x_name == "x" else (R, H)
    for t, n, dt, sh in ((x_src, x_name, torch.bfloat16, x_shape), (h_perm, "h_perm", torch.bfloat16, (R, I)),
                         (topk_w, "topk_w", torch.float32, (T, k)), (m_indptr, "m_indptr", torch.int32, (E + 1,)),
                         (row_to_slot, "row_to_slot", torch.int32, (R,)),
                         (slot_to_row, "slot_to_row", torch.int32, (R,)), (w_perm, "w_perm", torch.float32, (R,)),
                         (w_gate_up, "w_gate_up", torch.bfloat16, (E, nin, H)),
                         (w_down, "w_down", torch.bfloat16, (E, H, I))):
        _need(t, n, dt, sh)
    if gu_perm is not None:
        _need(gu_perm, "gu_perm", torch.float32, (R, nin))
    dev = dy.device
    out = dict(out or {})
    dx = _out(out.get("dx"), "dx", torch.bfloat16, (T, H), dev)
    dwgu = _out(out.get("dw_gate_up"), "dw_gate_up", torch.bfloat16, (E, nin, H), dev)
    dwd = _out(out.get("dw_down"), "dw_down", torch.bfloat16, (E, H, I), dev)
    dl = _out(out.get("d_logits"), "d_logits", torch.float32, (T, E), dev)
    ws = _workspace(workspace, workspace_bytes("bwd_dx_dw", T=T, H=H, I=I, E=E, k=k, saved_gu=gu_perm is not None,
                                               gather=x_name == "x"), dev)
    n = ctypes.c_size_t(ws.numel())
    extra = () if act is None else (_act_id(act[0]), float(act[1]))
    _check(fn, getattr(lib, fn)(
        _ptr(dy), _ptr(x_src), _ptr(h_perm), _ptr(gu_perm), _ptr(topk_ids), _ptr(topk_w), _ptr(m_indptr),
        _ptr(row_to_slot), _ptr(slot_to_row), _ptr(w_perm), _ptr(w_gate_up), _ptr(w_down), T, H, I, E, k, *extra,
        _ptr(dx), _ptr(dwgu), _ptr(dwd), _ptr(dl), _ptr(ws), ctypes.byref(n), _stream(stream)))
    return dx, dwgu, dwd, dl


def bwd_dx_dw(dy, x_perm, h_perm, gu_perm, topk_ids, topk_w, m_indptr, row_to_slot, slot_to_row, w_perm, w_gate_up,
              w_down, *, out=None, workspace=None, stream=None):
    """Backward of the layer: returns (dx [T,H], dw_gate_up [E,2I,H], dw_down [E,H,I], d_logits [T,E])."""
    return _bwd("liger_moe_bwd_dx_dw", dy, x_perm, "x_perm", h_perm, gu_perm, topk_ids, topk_w, m_indptr,
                row_to_slot, slot_to_row, w_perm, w_gate_up, w_down, out, workspace, stream)


def bwd_dx_dw_glu(dy, x_perm, h_perm, gu_perm, topk_ids, topk_w, m_indptr, row_to_slot, slot_to_row, w_perm,
                  w_gate_up, w_down, activation="swiglu", clamp=0.0, *, out=None, workspace=None, stream=None):
    """bwd_dx_dw for a forward with another activation (needed when gu_perm is None: the
    derivative factors are recomputed with that activation; always for relu2, whose w_gate_up is
    the up weight [E, I, H], gu_perm [R, I] and dw_gate_up [E, I, H])."""
    return _bwd("liger_moe_bwd_dx_dw_glu", dy, x_perm, "x_perm", h_perm, gu_perm, topk_ids, topk_w, m_indptr,
                row_to_slot, slot_to_row, w_perm, w_gate_up, w_down, out, workspace, stream, act=(activation, clamp))


def bwd_dx_dw_gather(dy, x, h_perm, gu_perm, topk_ids, topk_w, m_indptr, row_to_slot, slot_to_row, w_perm,
                     w_gate_up, w_down, *, out=None, workspace=None, stream=None):
    """The backward on token-major x [T,H] (no x_perm); same outputs as bwd_dx_dw."""
    return _bwd("liger_moe_bwd_dx_dw_gather", dy, x, "x", h_perm, gu_perm, topk_ids, topk_w, m_indptr,
                row_to_slot, slot_to_row, w_perm, w_gate_up, w_down, out, workspace, stream)


def selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Runs the bounded-wait self-test: a wait that nothing completes gives up after limit_us and
    sets the WAIT_TIMEOUT bit, which device_error() then returns."""
    lib = load_library()
    _check("liger_moe_selftest_wait_timeout", lib.liger_moe_selftest_wait_timeout(int(limit_us), _stream(stream)))


def device_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error bits (0 = none)."""
    lib = load_library()
    flags = ctypes.c_int(0)
    rc = lib.liger_moe_device_error(_stream(stream), ctypes.byref(flags))
    if rc not in (OK, -6):
        _check("liger_moe_device_error", rc)
    return flags.value


def set_dw_fp16(on: bool = True) -> None:
    """Heavy experts' weight gradients in one fp16 pass (True, the default) or as bf16 hi + lo parts."""
    _check("liger_moe_set_dw_fp16", load_library().liger_moe_set_dw_fp16(1 if on else 0))


def trace_enable(on: bool = True) -> None:
    """Turns the library's per-kernel CUDA-event trace on or off (clears the log)."""
    _check("liger_moe_trace_enable", load_library().liger_moe_trace_enable(1 if on else 0))


def trace_launch_counts() -> list[int]:
    """Kernel launches of every logged interval (one, or two for a GEMM split in two launches)."""
    lib = load_library()
    out = []
    n = ctypes.c_int()
    for i in range(lib.liger_moe_trace_count()):
        _check("liger_moe_trace_launches", lib.liger_moe_trace_launches(i, ctypes.byref(n)))
        out.append(int(n.value))
    return out


def trace_records() -> list[tuple[str, float]]:
    """(kernel name, device milliseconds) of every launch logged since trace_enable(True)."""
    lib = load_library()
    out = []
    name = ctypes.c_char_p()
    ms = ctypes.c_float()
    for i in range(lib.liger_moe_trace_count()):
        _check("liger_moe_trace_get", lib.liger_moe_trace_get(i, ctypes.byref(name), ctypes.byref(ms)))
        out.append((name.value.decode(), float(ms.value)))
    return out
