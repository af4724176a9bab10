"""GPU parity of the router and the dispatch against the oracle (bit-exact integers)."""
import numpy as np
import pytest
import torch

import mixture_experts_routed_router_gb300 as moe
import oracle
import synthetic
from tests.gpu_util import to_dev, to_host

pytestmark = pytest.mark.gpu


def _logits(T, E, seed, kind="normal"):
    rng = np.random.default_rng(seed)
    l = rng.standard_normal((T, E)).astype(np.float32)
    if kind == "ties":
        l = np.round(l * 2.0) / 2.0
    elif kind == "special":
        l[:, ::7] = 0.0
        l[:, 3::11] = -0.0
        l[::5, 1] = np.nan
        l[::3, 2] = np.inf
        l[1::4, 4] = -np.inf
    return l


@pytest.mark.parametrize("T,E,k", [(256, 8, 2), (50, 37, 5), (1000, 256, 8), (333, 512, 10), (64, 128, 8),
                                   (17, 1024, 32), (9, 32, 32), (1, 3, 2), (5, 1, 1), (129, 33, 1)])
@pytest.mark.parametrize("kind", ["normal", "ties"])
def test_route_topk_bit_exact_ids(T, E, k, kind):
    l = _logits(T, E, seed=T * 7 + E, kind=kind)
    ids, w = moe.route_topk(to_dev(l), k)
    ref_ids, ref_w = oracle.route_topk(l, k)
    np.testing.assert_array_equal(to_host(ids), ref_ids)
    np.testing.assert_allclose(to_host(w), ref_w, rtol=2e-6, atol=1e-8)
    assert moe.device_error() == 0


def test_route_topk_special_values():
    l = _logits(200, 64, seed=3, kind="special")
    ids, _ = moe.route_topk(to_dev(l), 6)
    ref_ids, _ = oracle.route_topk(l, 6)
    np.testing.assert_array_equal(to_host(ids), ref_ids)


def test_route_topk_zero_tokens():
    ids, w = moe.route_topk(torch.empty((0, 16), dtype=torch.float32, device="cuda"), 4)
    assert ids.shape == (0, 4) and w.shape == (0, 4)


def _ids_from(T, E, k, seed, skew=0.0):
    rng = np.random.default_rng(seed)
    p = np.exp(-skew * np.arange(E))
    p /= p.sum()
    return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,H,E,k,skew", [(256, 256, 8, 2, 0.0), (300, 64, 37, 5, 0.3), (1000, 128, 256, 8, 0.0),
                                          (700, 320, 5, 3, 0.0), (64, 4096, 128, 8, 0.0), (2049, 64, 512, 10, 0.05),
                                          (3, 64, 16, 2, 0.0), (1, 64, 1, 1, 0.0)])
def test_dispatch_bit_exact(T, H, E, k, skew):
    ids = _ids_from(T, E, k, seed=T + E, skew=skew)
    rng = np.random.default_rng(5)
    w = rng.random((T, k), dtype=np.float32)
    x = synthetic.normal_bf16((T, H), seed=1, stream=11, sigma=1.0)
    d = moe.dispatch(to_dev(ids), to_dev(w), to_dev(x), E)
    ref = oracle.dispatch(ids, w, x, E)
    for key in ("counts", "m_indptr", "row_to_slot", "slot_to_row", "w_perm", "x_perm"):
        np.testing.assert_array_equal(to_host(d[key]), ref[key], err_msg=key)
    assert moe.device_error() == 0


def test_dispatch_is_deterministic_across_calls():
    ids = _ids_from(4096, 64, 8, seed=9)
    a = moe.dispatch(to_dev(ids), None, None, 64)
    b = moe.dispatch(to_dev(ids), None, None, 64)
    for key in ("counts", "m_indptr", "row_to_slot", "slot_to_row"):
        assert torch.equal(a[key], b[key])


def test_dispatch_empty_experts_and_zero_tokens():
    ids = np.array([[3, 1], [1, 3], [5, 1]], np.int32)
    d = moe.dispatch(to_dev(ids), None, None, 9)
    ref = oracle.dispatch(ids, None, None, 9)
    for key in ("counts", "m_indptr", "row_to_slot", "slot_to_row"):
        np.testing.assert_array_equal(to_host(d[key]), ref[key])
    d0 = moe.dispatch(torch.empty((0, 2), dtype=torch.int32, device="cuda"), None, None, 7)
    assert to_host(d0["m_indptr"]).tolist() == [0] * 8
    assert to_host(d0["counts"]).tolist() == [0] * 7


def test_dispatch_flags_out_of_range_expert_ids():
    ids = np.array([[0, 1], [2, 9], [1, 0]], np.int32)  # 9 is outside [0, 4)
    moe.dispatch(to_dev(ids), None, None, 4)
    assert moe.device_error() & 0x1
    assert moe.device_error() == 0  # reading clears the flag
