"""liger_moe_dispatch_noalloc (the dispatch for callers that cannot allocate) against liger_moe_dispatch.

Callers with no way to allocate device memory (fixed memory plans, plug-ins that
only see their own tensors) use this entry point; its scratch is a fixed array in
the library.  The test calls both entry points through the C ABI on the same
inputs, twice in a row (the second call reuses the array the first one left
behind), and requires identical outputs: every output is integer or a copy, so
the tolerance is exact equality.
"""
import ctypes

import numpy as np
import pytest
import torch

import mixture_experts_routed_router_gb300 as moe
import synthetic

pytestmark = pytest.mark.gpu


def _lib():
    lib = moe.load_library()
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.liger_moe_dispatch_noalloc.argtypes = [P, P, P, I, I, I, I, P, P, P, P, P, P, P]
    lib.liger_moe_dispatch_noalloc.restype = ctypes.c_int
    return lib


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, ids, w, x, E):
    T, k = ids.shape
    R, H = T * k, x.shape[1]
    o = dict(counts=torch.empty(E, dtype=torch.int32, device="cuda"),
             m_indptr=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
             row_to_slot=torch.empty(R, dtype=torch.int32, device="cuda"),
             slot_to_row=torch.empty(R, dtype=torch.int32, device="cuda"),
             w_perm=torch.empty(R, dtype=torch.float32, device="cuda"),
             x_perm=torch.empty((R, H), dtype=torch.bfloat16, device="cuda"))
    rc = lib.liger_moe_dispatch_noalloc(_ptr(ids), _ptr(w), _ptr(x), T, H, E, k, _ptr(o["counts"]),
                                        _ptr(o["m_indptr"]), _ptr(o["row_to_slot"]), _ptr(o["slot_to_row"]),
                                        _ptr(o["w_perm"]), _ptr(o["x_perm"]),
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, moe.load_library().liger_moe_last_cuda_error()
    return o


@pytest.mark.parametrize("name", ["fwd_T8192_H2048_I512_E256_k8", "tiny_T256_H256_I128_E8_k2"])
def test_noalloc_dispatch_matches_dispatch_twice(name):
    lib = _lib()
    wl = synthetic.WORKLOADS[name]
    inp = synthetic.make_inputs(wl, want=("x", "logits"))
    logits = torch.from_numpy(inp["logits"]).cuda()
    x = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).cuda()
    ids, w = moe.route_topk(logits, wl.k)
    ref = moe.dispatch(ids, w, x, wl.E)
    for _ in range(2):
        got = _noalloc(lib, ids, w, x, wl.E)
        torch.cuda.synchronize()
        assert moe.device_error() == 0
        for key in ("counts", "m_indptr", "row_to_slot", "slot_to_row", "w_perm", "x_perm"):
            assert torch.equal(got[key], ref[key]), key


def test_noalloc_dispatch_rejects_sizes_beyond_its_scratch():
    lib = _lib()
    T, E, k = 65536, 1024, 8  # ceil(T*k/256) * E * 4 bytes = 8 MiB > 1 MiB
    d = ctypes.c_void_p(256)  # never dereferenced: the call is rejected before any launch
    assert lib.liger_moe_dispatch_noalloc(d, None, None, T, 0, E, k, d, d, d, d, None, None, None) == -3
