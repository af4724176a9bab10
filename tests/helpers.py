"""Shared test utilities: the error metrics and an fp64 dense restatement of the layer.

The dense restatement is deliberately different from the oracle's per-token
loops: it evaluates every expert on every token with ``torch.einsum`` in
float64 and masks the result with the dense gate matrix G[t, e] (zero off the
selected k).  It is the brute-force check the oracle is pinned against; it
calls nothing in ``oracle/``.
"""
from __future__ import annotations

import numpy as np
import torch

# Pass bar of the CUDA path against the oracle, per output tensor.
MAX_REL_TOL = 2e-2
MEAN_REL_TOL = 1e-2


def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rel_errors(got, ref) -> tuple[float, float]:
    """(max_rel, mean_rel) of ``got`` against ``ref``.

    max_rel  = max_i |g_i - r_i| / max(|r_i|, rms(r))   (floor at rms keeps near-zero
               entries from dominating)
    mean_rel = sum |g - r| / sum |r|
    """
    g = np.asarray(got, dtype=np.float64).ravel()
    r = np.asarray(ref, dtype=np.float64).ravel()
    if r.size == 0:
        return 0.0, 0.0
    d = np.abs(g - r)
    if not np.all(np.isfinite(d)):
        return float("inf"), float("inf")
    rms = float(np.sqrt(np.mean(r * r)))
    s = float(np.sum(np.abs(r)))
    if s == 0.0:
        m = float(d.max())
        return m, m
    denom = np.maximum(np.abs(r), rms)
    return float(np.max(d / denom)), float(np.sum(d) / s)


def rel_errors_per_expert(got, ref) -> tuple[float, float]:
    """Metrics for weight gradients [E, ...]: max_rel uses each expert's own rms as the floor.

    Expert gradients differ in scale by the square root of their row counts
    (strongly so under skewed routing), so one tensor-wide rms floor would
    measure a heavy expert's near-zero entries against a light expert's scale.
    mean_rel stays tensor-wide.
    """
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    mx = max((rel_errors(g[e], r[e])[0] for e in range(r.shape[0])), default=0.0)
    return mx, rel_errors(g, r)[1]


def assert_close(got, ref, name, max_rel=MAX_REL_TOL, mean_rel=MEAN_REL_TOL, per_expert=False):
    mx, mn = (rel_errors_per_expert if per_expert else rel_errors)(got, ref)
    assert mx <= max_rel and mn <= mean_rel, f"{name}: max_rel={mx:.3e} (tol {max_rel}) mean_rel={mn:.3e} (tol {mean_rel})"
    return mx, mn


def off_selection(ids: np.ndarray, E: int) -> np.ndarray:
    """[T, E] mask, True where expert e is not among token t's selected ids (where d_logits must
    be exactly zero).  Taken from the routing itself: a selected entry may be zero too."""
    ids = np.asarray(ids, dtype=np.int64)
    mask = np.ones((ids.shape[0], E), dtype=bool)
    np.put_along_axis(mask, ids, False, axis=1)
    return mask


def topk_bruteforce(logits: np.ndarray, k: int) -> np.ndarray:
    """Selected experts per token: full sort by (logit descending, id ascending)."""
    T, E = logits.shape
    out = np.empty((T, k), np.int32)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))
        out[t] = order[:k]
    return out


def gated_act_torch(g, u, act="swiglu", clamp=0.0):
    """The gated activations in plain torch ops (independent of the oracle's C++):
    swiglu silu(g) u; swiglu_bounded silu(min(g, c)) clamp(u, -c, c); swiglu_oai
    gc sigmoid(1.702 gc) (clamp(u, -c, c) + 1) with gc = min(g, c); geglu gelu_tanh(g) u;
    reglu relu(g) u.  torch.clamp passes gradient on the closed interval."""
    F = torch.nn.functional
    if act == "swiglu":
        return F.silu(g) * u
    if act == "swiglu_bounded":
        return F.silu(torch.clamp(g, max=clamp)) * torch.clamp(u, -clamp, clamp)
    if act == "swiglu_oai":
        gc = torch.clamp(g, max=clamp)
        return gc * torch.sigmoid(1.702 * gc) * (torch.clamp(u, -clamp, clamp) + 1.0)
    if act == "geglu":
        return F.gelu(g, approximate="tanh") * u
    if act == "reglu":
        return F.relu(g) * u
    raise ValueError(act)


def dense_layer_fp64(x_bits, wgu_bits, wd_bits, logits, sel, requires_grad=False, act="swiglu", clamp=0.0):
    """fp64 dense evaluation of the routed SwiGLU layer (or another activation: gated_act_torch;
    relu2 takes the up weight [E, I, H] as wgu and h = relu(x Wup^T)^2).

    Y[t, c] = sum_e G[t, e] * sum_n silu(g[t,e,n]) * u[t,e,n] * Wd[e, c, n]
    with g = x Wgu[e, :I]^T, u = x Wgu[e, I:]^T and G = softmax over the
    selected logits (zero elsewhere).  Returns (Y, leaves) with leaves the
    tensors gradients can be taken against (x, wgu, wd, logits).
    """
    x = torch.tensor(bf16_to_f64(x_bits), requires_grad=requires_grad)
    wgu = torch.tensor(bf16_to_f64(wgu_bits), requires_grad=requires_grad)
    wd = torch.tensor(bf16_to_f64(wd_bits), requires_grad=requires_grad)
    lg = torch.tensor(np.asarray(logits, dtype=np.float64), requires_grad=requires_grad)
    T, E = lg.shape
    I = wgu.shape[1] // 2 if act != "relu2" else wgu.shape[1]
    mask = torch.zeros((T, E), dtype=torch.bool)
    mask[torch.arange(T)[:, None], torch.tensor(sel, dtype=torch.long)] = True
    G = torch.softmax(lg.masked_fill(~mask, float("-inf")), dim=1)
    if act == "relu2":  # not gated: wgu is the up weight [E, I, H], h = relu(x Wup^T)^2
        a = torch.relu(torch.einsum("th,enh->ten", x, wgu)) ** 2
    else:
        gu = torch.einsum("th,enh->ten", x, wgu)
        a = gated_act_torch(gu[..., :I], gu[..., I:], act, clamp)
    o = torch.einsum("ten,ecn->tec", a, wd)
    Y = torch.einsum("te,tec->tc", G, o)
    return Y, dict(x=x, wgu=wgu, wd=wd, logits=lg, G=G)


def dense_swiglu_mlp_fp64(x_bits, wgu_e_bits, wd_e_bits):
    """One dense SwiGLU MLP, down(silu(gate x) * up x), in fp64 (Liger's SwiGLU MLP form)."""
    x = torch.tensor(bf16_to_f64(x_bits))
    wgu = torch.tensor(bf16_to_f64(wgu_e_bits))
    wd = torch.tensor(bf16_to_f64(wd_e_bits))
    I = wgu.shape[0] // 2
    gate = x @ wgu[:I].T
    up = x @ wgu[I:].T
    return (torch.nn.functional.silu(gate) * up) @ wd.T


def swiglu_factors(gu_f32: np.ndarray) -> np.ndarray:
    """SwiGLU derivative factors [dh/dg | dh/du] of h = silu(g) u from [g | u] (float32 out).

    dh/dg = u s (1 + g (1 - s)), dh/du = silu(g) = g s, with s = 1 / (1 + exp(-g)).
    """
    gu = np.asarray(gu_f32, dtype=np.float64)
    I = gu.shape[1] // 2
    g, u = gu[:, :I], gu[:, I:]
    s = 1.0 / (1.0 + np.exp(-g))
    return np.concatenate([u * s * (1.0 + g * (1.0 - s)), g * s], axis=1).astype(np.float32)
