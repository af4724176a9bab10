"""Pins for the oracle's deterministic expert-major dispatch, CPU only.

LightMoE README, "MoE training" / "Grouped GEMM": expert-major contiguous rows,
m_indptr (E+1, int32), permuted routing weights, inverse slots; zero-row
experts valid.  Reading: rows of one expert are in slot order (stable sort).
"""
import numpy as np
import pytest

import oracle
import synthetic


def _ids(T, E, k, seed, skew=0.0):
    rng = np.random.default_rng(seed)
    p = np.exp(-skew * np.arange(E))
    p /= p.sum()
    out = np.empty((T, k), np.int32)
    for t in range(T):
        out[t] = rng.choice(E, size=k, replace=False, p=p)
    return out


@pytest.mark.parametrize("T,E,k,skew", [(256, 8, 2, 0.0), (300, 37, 5, 0.3), (129, 64, 8, 0.0),
                                        (64, 128, 8, 1.0), (1, 4, 4, 0.0)])
def test_matches_stable_argsort(T, E, k, skew):
    ids = _ids(T, E, k, seed=T + E, skew=skew)
    rng = np.random.default_rng(1)
    w = rng.random((T, k), dtype=np.float32)
    x = rng.integers(0, 2 ** 16, size=(T, 64), dtype=np.uint16)
    d = oracle.dispatch(ids, w, x, E)
    flat = ids.ravel()
    ref_r2s = np.argsort(flat, kind="stable").astype(np.int32)  # library stable sort
    np.testing.assert_array_equal(d["row_to_slot"], ref_r2s)
    np.testing.assert_array_equal(d["counts"], np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(d["m_indptr"], np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    s2r = np.empty_like(ref_r2s)
    s2r[ref_r2s] = np.arange(T * k, dtype=np.int32)
    np.testing.assert_array_equal(d["slot_to_row"], s2r)
    np.testing.assert_array_equal(d["w_perm"], w.ravel()[ref_r2s])
    np.testing.assert_array_equal(d["x_perm"], x[ref_r2s // k])


def test_invariants_on_synthetic_routing():
    wl = synthetic.WORKLOADS["tiny_T256_H256_I128_E8_k2"]
    inp = synthetic.make_inputs(wl, want=("x", "logits"))
    ids, w = oracle.route_topk(inp["logits"], wl.k)
    d = oracle.dispatch(ids, w, inp["x"], wl.E)
    R = wl.T * wl.k
    assert d["counts"].sum() == R
    assert d["m_indptr"][-1] == R
    np.testing.assert_array_equal(d["slot_to_row"][d["row_to_slot"]], np.arange(R))
    np.testing.assert_array_equal(d["row_to_slot"][d["slot_to_row"]], np.arange(R))
    for e in range(wl.E):
        rows = d["row_to_slot"][d["m_indptr"][e]:d["m_indptr"][e + 1]]
        assert np.all(ids.ravel()[rows] == e)
        assert np.all(np.diff(rows // wl.k) > 0)  # tokens strictly ascending within an expert


def test_empty_experts_and_zero_tokens():
    ids = np.array([[3, 1], [1, 3]], np.int32)
    d = oracle.dispatch(ids, None, None, 6)
    np.testing.assert_array_equal(d["counts"], [0, 2, 0, 2, 0, 0])
    np.testing.assert_array_equal(d["m_indptr"], [0, 0, 2, 2, 4, 4, 4])
    np.testing.assert_array_equal(d["row_to_slot"], [1, 2, 0, 3])
    d0 = oracle.dispatch(np.zeros((0, 2), np.int32), None, None, 5)
    np.testing.assert_array_equal(d0["m_indptr"], np.zeros(6))


def test_out_of_range_id_is_rejected():
    with pytest.raises(ValueError):
        oracle.dispatch(np.array([[0, 7]], np.int32), None, None, 4)
