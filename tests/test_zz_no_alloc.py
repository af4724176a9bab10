"""liger_moe_dispatch_noalloc (the dispatch for callers that cannot allocate) against the oracle and liger_moe_dispatch.

Callers with no way to allocate device memory (fixed memory plans, plug-ins that
only see their own tensors) use this entry point; its scratch is a fixed array in
the library.  The test calls it through the C ABI twice in a row on the same
inputs (the second call reuses the array the first one left behind) and requires
the oracle's dispatch bit for bit, and the same bytes as liger_moe_dispatch
(whose x_perm copy is the reference for the row copy): every output is integer
or a copy, so the tolerance is exact equality.  It runs at the largest size the
array accepts (T*k = 131072 at E = 512, where the histograms fill it exactly)
and checks that a size one slot past it is refused, and that a call leaves the
device's free memory unchanged.
"""
import ctypes

import numpy as np
import pytest
import torch

import mixture_experts_routed_router_gb300 as moe
import oracle
import synthetic

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 1 << 20  # the array's stated size


def _lib():
    lib = moe.load_library()
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.liger_moe_dispatch_noalloc.argtypes = [P, P, P, I, I, I, I, P, P, P, P, P, P, P]
    lib.liger_moe_dispatch_noalloc.restype = ctypes.c_int
    return lib


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _outputs(T, k, H, E):
    R = T * k
    return dict(counts=torch.empty(E, dtype=torch.int32, device="cuda"),
                m_indptr=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
                row_to_slot=torch.empty(R, dtype=torch.int32, device="cuda"),
                slot_to_row=torch.empty(R, dtype=torch.int32, device="cuda"),
                w_perm=torch.empty(R, dtype=torch.float32, device="cuda"),
                x_perm=torch.empty((R, H), dtype=torch.bfloat16, device="cuda"))


def _noalloc(lib, ids, w, x, E, o):
    T, k = ids.shape
    H = x.shape[1]
    for v in o.values():  # stale bytes from an earlier call must not survive
        v.fill_(-1 if v.dtype != torch.bfloat16 else 0)
    rc = lib.liger_moe_dispatch_noalloc(_ptr(ids), _ptr(w), _ptr(x), T, H, E, k, _ptr(o["counts"]),
                                        _ptr(o["m_indptr"]), _ptr(o["row_to_slot"]), _ptr(o["slot_to_row"]),
                                        _ptr(o["w_perm"]), _ptr(o["x_perm"]),
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, moe.load_library().liger_moe_last_cuda_error()
    return o


@pytest.mark.parametrize("name", ["fwd_T8192_H2048_I512_E256_k8", "tiny_T256_H256_I128_E8_k2",
                                  "edge_T16384_H64_I64_E512_k8"])
def test_noalloc_dispatch_matches_oracle_twice(name):
    lib = _lib()
    wl = synthetic.workload(name)
    if name.startswith("edge"):  # the histograms fill the array exactly
        assert -(-wl.R // 256) * wl.E * 4 == SCRATCH_BYTES
    inp = synthetic.make_inputs(wl, want=("x", "logits"))
    logits = torch.from_numpy(inp["logits"]).cuda()
    x = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).cuda()
    ids, w = moe.route_topk(logits, wl.k)
    rids, rw = oracle.route_topk(inp["logits"], wl.k)
    np.testing.assert_array_equal(ids.cpu().numpy(), rids)
    ref = oracle.dispatch(rids, rw, None, wl.E)
    lib_ref = moe.dispatch(ids, w, x, wl.E)
    o = _outputs(wl.T, wl.k, wl.H, wl.E)
    for call in range(2):
        free0 = torch.cuda.mem_get_info()[0] if call == 1 else None
        got = _noalloc(lib, ids, w, x, wl.E, o)
        torch.cuda.synchronize()
        if call == 1:
            assert torch.cuda.mem_get_info()[0] == free0, "the call changed the device's free memory"
        assert moe.device_error() == 0
        for key in ("counts", "m_indptr", "row_to_slot", "slot_to_row"):
            np.testing.assert_array_equal(got[key].cpu().numpy(), ref[key], err_msg=f"{key} (call {call})")
        # w_perm is topk_w of each row's slot (a copy); x_perm the token rows (a copy)
        np.testing.assert_array_equal(got["w_perm"].cpu().numpy(), w.cpu().numpy().ravel()[ref["row_to_slot"]])
        for key in ("counts", "m_indptr", "row_to_slot", "slot_to_row", "w_perm", "x_perm"):
            assert torch.equal(got[key], lib_ref[key]), f"{key} (call {call})"


def test_noalloc_dispatch_rejects_sizes_beyond_its_scratch():
    lib = _lib()
    d = ctypes.c_void_p(256)  # never dereferenced: the call is rejected before any launch
    # one slot past the largest accepted size at E = 512: 513 chunks x 512 experts x 4 bytes > 1 MiB
    assert lib.liger_moe_dispatch_noalloc(d, None, None, 131073, 0, 512, 1, d, d, d, d, None, None, None) == -3
    T, E, k = 65536, 1024, 8  # ceil(T*k/256) * E * 4 bytes = 8 MiB
    assert lib.liger_moe_dispatch_noalloc(d, None, None, T, 0, E, k, d, d, d, d, None, None, None) == -3
