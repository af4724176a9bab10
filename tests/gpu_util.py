"""Moving test inputs between numpy (bf16 as uint16 bits) and CUDA tensors; the library's
process-wide weight-gradient precision switch as a context manager."""
import contextlib

import numpy as np
import torch

import mixture_experts_routed_router_gb300 as moe


@contextlib.contextmanager
def dw_fp16(on: bool):
    """Heavy experts' weight gradients in one fp16 pass (on) or as bf16 hi + lo parts, restoring the default."""
    moe.set_dw_fp16(on)
    try:
        yield
    finally:
        moe.set_dw_fp16(True)


def to_dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    t = torch.from_numpy(a).cuda()
    return t if dtype is None else t.to(dtype)


def to_host(t: torch.Tensor) -> np.ndarray:
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()
