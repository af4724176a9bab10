"""Seeded synthetic inputs for the routed MoE layer (no step of the layer lives here).

Workloads follow the shapes the pages give for the routed SwiGLU MoE layer
(LightMoE README, "Compatibility" model-contract table; LigerCute README,
"MoE performance": D=2048, I=768, E=128, K=8 at 8,192 tokens).  Values:

* ``x[T,H]``       = bf16(N(0, 1))
* ``Wr[E,H]``      = bf16(N(0, 0.02))            router projection (upstream of the layer)
* ``logits[T,E]``  = float(sum_h x*Wr + bias)    summed in double, rounded once
* ``bias[e]``      = -s * ln(pi(e) + 1)          only for the Zipf(s) workload, pi a seeded
                                                 permutation (log of an unnormalised Zipf pmf)
* ``W_gu[E,2I,H]`` = bf16(N(0, 1/sqrt(H)))       rows [0,I) gate, [I,2I) up
* ``W_d[E,H,I]``   = bf16(N(0, 1/sqrt(I)))
* ``dY[T,H]``      = bf16(N(0, 1))               upstream gradient

Every tensor has its own counter-based stream (see ``gen.c``), so any tensor
can be regenerated alone and the fill does not depend on the thread count.
bf16 tensors are returned as ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

STREAM_X, STREAM_WR, STREAM_WGU, STREAM_WD, STREAM_DY, STREAM_PERM = 1, 2, 3, 4, 5, 6


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    zipf_s: float | None = None
    router_std: float = 0.02

    @property
    def R(self) -> int:
        return self.T * self.k

    def as_dict(self) -> dict:
        d = dict(workload=self.name, T=self.T, H=self.H, I=self.I, E=self.E, k=self.k)
        if self.zipf_s is not None:
            d["router_bias"] = f"zipf(s={self.zipf_s})"
        return d


WORKLOADS = {
    w.name: w
    for w in (
        Workload("tiny_T256_H256_I128_E8_k2", 256, 256, 128, 8, 2),
        Workload("fwd_T8192_H2048_I512_E256_k8", 8192, 2048, 512, 256, 8),
        Workload("fwd_zipf_T8192_H4096_I1024_E512_k10", 8192, 4096, 1024, 512, 10, zipf_s=1.2),
        Workload("decode_T64_H4096_I1536_E128_k8", 64, 4096, 1536, 128, 8),
        Workload("train_T8192_H2048_I768_E128_k8", 8192, 2048, 768, 128, 8),
    )
}


def workload(name: str) -> Workload:
    """A named workload, or one spelled out as <label>_T<T>_H<H>_I<I>_E<E>_k<k>[_zipf<s>]."""
    if name in WORKLOADS:
        return WORKLOADS[name]
    import re

    m = re.fullmatch(r"[A-Za-z0-9]+_T(\d+)_H(\d+)_I(\d+)_E(\d+)_k(\d+)(?:_zipf([0-9.]+))?", name)
    if not m:
        raise KeyError(f"unknown workload {name!r}")
    T, H, I, E, k = (int(v) for v in m.groups()[:5])
    return Workload(name, T, H, I, E, k, zipf_s=float(m.group(6)) if m.group(6) else None)


def build(force: bool = False) -> str:
    """Compile gen.c into libsynth.so beside it (gcc, no vendor code)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = f"{_LIB_PATH}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.synth_normal_bf16.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint64,
                                              ctypes.c_uint64, ctypes.c_double, ctypes.c_int]
            lib.synth_permutation.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64,
                                              ctypes.c_uint64]
            lib.synth_router_logits.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_void_p, ctypes.c_int]
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_bf16(shape, seed: int, stream: int, sigma: float) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    _load().synth_normal_bf16(out.ctypes.data, out.size, seed, stream, float(sigma), _threads())
    return out


def permutation(n: int, seed: int, stream: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _load().synth_permutation(out.ctypes.data, n, seed, stream)
    return out


def router_logits(x: np.ndarray, wr: np.ndarray, bias: np.ndarray | None) -> np.ndarray:
    T, H = x.shape
    E = wr.shape[0]
    x = np.ascontiguousarray(x, dtype=np.uint16)
    wr = np.ascontiguousarray(wr, dtype=np.uint16)
    out = np.empty((T, E), dtype=np.float32)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float64)
    _load().synth_router_logits(x.ctypes.data, wr.ctypes.data, None if b is None else b.ctypes.data,
                                T, H, E, out.ctypes.data, _threads())
    return out


def zipf_bias(E: int, s: float, seed: int) -> np.ndarray:
    perm = permutation(E, seed, STREAM_PERM).astype(np.float64)
    return -s * np.log(perm + 1.0)


def make_inputs(w: Workload, seed: int = 0, want=("x", "logits", "wgu", "wd", "dy")) -> dict:
    """All inputs of one workload as numpy arrays (bf16 as uint16 bits).  ``"wr"`` in ``want``
    adds the router weight ``wr`` and bias ``bias`` (float32 [E], or None without a Zipf skew)."""
    out: dict = {}
    need_x = "x" in want or "logits" in want
    if need_x:
        out["x"] = normal_bf16((w.T, w.H), seed, STREAM_X, 1.0)
    if "logits" in want or "wr" in want:
        wr = normal_bf16((w.E, w.H), seed, STREAM_WR, w.router_std)
        bias = zipf_bias(w.E, w.zipf_s, seed) if w.zipf_s is not None else None
        if "logits" in want:
            out["logits"] = router_logits(out["x"], wr, bias)
        if "wr" in want:  # the router weight and (Zipf workload) bias themselves, as inputs
            out["wr"] = wr
            out["bias"] = None if bias is None else bias.astype(np.float32)
    if "wgu" in want:
        out["wgu"] = normal_bf16((w.E, 2 * w.I, w.H), seed, STREAM_WGU, 1.0 / math.sqrt(w.H))
    if "wd" in want:
        out["wd"] = normal_bf16((w.E, w.H, w.I), seed, STREAM_WD, 1.0 / math.sqrt(w.I))
    if "dy" in want:
        out["dy"] = normal_bf16((w.T, w.H), seed, STREAM_DY, 1.0)
    if "x" not in want:
        out.pop("x", None)
    return out


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 values exactly."""
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest even (finite values)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)
