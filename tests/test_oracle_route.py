"""Pins for the oracle's router (top-k + renormalised softmax), CPU only.

Routing reading (LightMoE README, "MoE inference" / "MoE training"): the k
largest logits per token, ties to the lower expert id, weights = softmax over
the selected k (= full softmax, top-k, renormalise).
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import topk_bruteforce

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_worked_example.json")


def _logits(T, E, seed, ties=False):
    rng = np.random.default_rng(seed)
    l = rng.standard_normal((T, E)).astype(np.float32)
    if ties:
        l = np.round(l * 2.0) / 2.0  # many exact ties
    return l


@pytest.mark.parametrize("T,E,k", [(64, 8, 2), (50, 37, 5), (33, 128, 8), (9, 512, 10), (5, 4, 4)])
@pytest.mark.parametrize("ties", [False, True])
def test_ids_match_bruteforce_sort(T, E, k, ties):
    l = _logits(T, E, seed=T * 1000 + E, ties=ties)
    ids, _ = oracle.route_topk(l, k)
    np.testing.assert_array_equal(ids, topk_bruteforce(l, k))


@pytest.mark.parametrize("T,E,k", [(64, 8, 2), (40, 64, 6), (7, 300, 12)])
def test_weights_are_renormalised_softmax(T, E, k):
    l = _logits(T, E, seed=7 + E)
    ids, w = oracle.route_topk(l, k)
    sel = np.take_along_axis(l.astype(np.float64), ids.astype(np.int64), axis=1)
    ref = torch.softmax(torch.tensor(sel), dim=1).numpy()
    np.testing.assert_allclose(w, ref, rtol=4e-7 * k, atol=1e-7)
    # renormalised gate weights sum to 1 within float rounding of k terms
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= k * 2.0 ** -23)
    # weights follow the selection order (non-increasing)
    assert np.all(np.diff(w, axis=1) <= 0)


def test_k1_weight_is_exactly_one():
    l = _logits(100, 16, seed=3)
    ids, w = oracle.route_topk(l, 1)
    assert np.all(w == 1.0)
    np.testing.assert_array_equal(ids[:, 0], np.argmax(l, axis=1))


def test_k_equals_E_is_full_softmax():
    l = _logits(20, 12, seed=4)
    ids, w = oracle.route_topk(l, 12)
    dense = np.zeros_like(l, dtype=np.float64)
    np.put_along_axis(dense, ids.astype(np.int64), w.astype(np.float64), axis=1)
    ref = torch.softmax(torch.tensor(l, dtype=torch.float64), dim=1).numpy()
    np.testing.assert_allclose(dense, ref, rtol=3e-6, atol=1e-8)
    # every expert appears exactly once per token
    assert np.all(np.sort(ids, axis=1) == np.arange(12))


def test_nan_logits_rank_last_and_ids_distinct():
    l = _logits(10, 16, seed=5)
    l[:, 3] = np.nan
    l[2, :] = np.nan
    ids, _ = oracle.route_topk(l, 4)
    assert not np.any(ids[np.arange(10) != 2] == 3)
    np.testing.assert_array_equal(ids[2], [0, 1, 2, 3])  # all NaN: by id
    for t in range(10):
        assert len(set(ids[t].tolist())) == 4


def test_closed_form_worked_example():
    g = json.load(open(GOLDEN))["routing"]
    ids, w = oracle.route_topk(np.array(g["logits"], np.float32), g["k"])
    np.testing.assert_array_equal(ids, np.array(g["ids"]))
    np.testing.assert_allclose(w, np.array(g["w"]), rtol=3e-7)
