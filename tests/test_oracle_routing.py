"""Pins of the oracle router (Eq. 2) against closed forms and brute force."""
import itertools

import numpy as np
import pytest

from oracle import routing


def test_softmax_closed_form(golden):
    g = golden("closed_forms.json")["softmax"]
    p = routing.softmax(np.array([g["logits"]], dtype=np.float32))[0]
    np.testing.assert_allclose(p, g["probs"], rtol=2e-7)


def test_topk_matches_brute_force_subset():
    rng = np.random.default_rng(0)
    T, Ne, k = 60, 7, 3
    logits = rng.standard_normal((T, Ne)).astype(np.float32)
    ids, gates = routing.route_topk(logits, k)
    p = np.exp(logits.astype(np.float64))
    p /= p.sum(1, keepdims=True)
    for t in range(T):
        best = max(itertools.combinations(range(Ne), k), key=lambda s: sum(logits[t, list(s)]))
        assert set(ids[t].tolist()) == set(best)
        # listed by descending logit
        assert all(logits[t, ids[t, j]] >= logits[t, ids[t, j + 1]] for j in range(k - 1))
        np.testing.assert_allclose(gates[t], p[t, ids[t]], rtol=1e-12)


def test_topk_ties_go_to_lower_id():
    logits = np.array([[1.0, 2.0, 2.0, 0.0], [5.0, 5.0, 5.0, 5.0]], dtype=np.float32)
    ids, _ = routing.route_topk(logits, 2)
    assert ids.tolist() == [[1, 2], [0, 1]]


def test_all_experts_chosen_when_k_equals_ne():
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((10, 5)).astype(np.float32)
    ids, gates = routing.route_topk(logits, 5)
    assert all(sorted(r) == list(range(5)) for r in ids.tolist())
    np.testing.assert_allclose(gates.sum(1), 1.0, rtol=1e-14)


def test_renorm_sums_to_one_and_keeps_ratios():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((20, 8)).astype(np.float32)
    ids, g0 = routing.route_topk(logits, 3)
    ids1, g1 = routing.route_topk(logits, 3, renorm=True)
    assert (ids == ids1).all()
    np.testing.assert_allclose(g1.sum(1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(g1[:, 1] / g1[:, 0], g0[:, 1] / g0[:, 0], rtol=1e-12)


def test_gate_matrix_is_eq2_topk_of_softmax():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((6, 5)).astype(np.float32)
    ids, gates = routing.route_topk(logits, 2)
    R = routing.gate_matrix(ids, gates, 5)
    p = routing.softmax(logits)
    for t in range(6):
        kth = np.sort(logits[t])[-2]
        for e in range(5):
            assert R[t, e] == (p[t, e] if logits[t, e] >= kth else 0.0)


def test_device_limited_closed_form(golden):
    g = golden("closed_forms.json")["device_limited"]
    ids, gates, kept, margin = routing.route_device_limited(
        np.array([g["logits"]], dtype=np.float32), g["top_k"], np.array(g["expert_to_vdev"]),
        2, g["n_keep"])
    assert ids[0].tolist() == g["ids"]
    np.testing.assert_allclose(gates[0], g["gates"], rtol=1e-15)
    assert kept[0].tolist() == [1]
    assert margin[0] > 0


def test_device_limited_keeping_all_devices_is_renormalised_topk():
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((30, 8)).astype(np.float32)
    e2v = np.array([0, 0, 1, 1, 2, 2, 3, 3])
    ids, gates, _, _ = routing.route_device_limited(logits, 3, e2v, 4, 4)
    ids2, gates2 = routing.route_topk(logits, 3, renorm=True)
    assert (ids == ids2).all()
    np.testing.assert_allclose(gates, gates2, rtol=1e-14)


def test_device_limited_stays_within_kept_devices():
    rng = np.random.default_rng(5)
    Ne, Nd, k, keep = 16, 8, 4, 2
    logits = rng.standard_normal((100, Ne)).astype(np.float32) * 2
    e2v = rng.permutation(np.repeat(np.arange(Nd), Ne // Nd))
    ids, gates, kept, _ = routing.route_device_limited(logits, k, e2v, Nd, keep)
    mass = routing.device_mass(logits, e2v, Nd)
    for t in range(100):
        assert len({int(e2v[e]) for e in ids[t]}) <= keep
        assert set(int(e2v[e]) for e in ids[t]) <= set(kept[t].tolist())
        # kept devices hold the largest masses
        assert min(mass[t, kept[t]]) >= max(np.delete(mass[t], kept[t]))
        np.testing.assert_allclose(gates[t].sum(), 1.0, rtol=1e-14)
