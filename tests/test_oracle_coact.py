"""Pins of the oracle co-activation graph (Eq. 3, 4), C_T (Eq. 5) and the
collaboration metrics (Sec. 3.2)."""
import numpy as np
import pytest

from oracle import coact, placement, routing


def test_worked_example(golden):
    g = golden("brim_worked_example.json")
    C = coact.coactivation(np.array(g["ids"]), g["n_experts"])
    assert C.tolist() == g["expect"]["coactivation"]
    P = coact.normalise(C)
    assert P.max() == 1.0 and P[0, 0] == 1.0 and P[1, 2] == 0.0


@pytest.mark.parametrize("seed,T,Ne,k", [(0, 100, 8, 2), (1, 257, 16, 5), (2, 64, 6, 6)])
def test_invariants(seed, T, Ne, k):
    rng = np.random.default_rng(seed)
    ids, _ = routing.route_topk(rng.standard_normal((T, Ne)).astype(np.float32), k)
    C = coact.coactivation(ids, Ne)
    assert (C == C.T).all()
    load = np.bincount(ids.ravel(), minlength=Ne)
    assert (np.diag(C) == load).all()
    assert np.trace(C) == T * k
    assert C.sum() - np.trace(C) == T * k * (k - 1)
    # brute force per pair
    for i in range(Ne):
        for j in range(Ne):
            assert C[i, j] == sum(1 for t in range(T) if i in ids[t] and j in ids[t])


@pytest.mark.parametrize("seed,Ne,Nd,k", [(3, 8, 4, 2), (4, 16, 4, 8), (5, 64, 16, 8),
                                          (6, 60, 4, 4), (7, 12, 12, 3)])
def test_ct_bounds_for_any_equal_placement(seed, Ne, Nd, k):
    rng = np.random.default_rng(seed)
    ids, _ = routing.route_topk(rng.standard_normal((300, Ne)).astype(np.float32), k)
    L = rng.permutation(Ne).reshape(Nd, Ne // Nd)
    ct = coact.replicas_per_token(ids, placement.expert_to_vdev(L))
    lo, hi = coact.ct_bounds(k, Ne, Nd)
    assert 1 <= lo <= hi
    assert ct.min() >= lo and ct.max() <= hi
    h = coact.ct_histogram(ct, hi)
    assert h.sum() == 300 and (h[:lo] == 0).all()


def test_single_device_ct_is_one():
    rng = np.random.default_rng(8)
    ids, _ = routing.route_topk(rng.standard_normal((50, 8)).astype(np.float32), 3)
    ct = coact.replicas_per_token(ids, np.zeros(8, dtype=int))
    assert (ct == 1).all()


def test_collaboration_metrics_by_hand():
    P = np.array([[1.0, 0.5, 0.1, 0.2],
                  [0.5, 1.0, 0.3, 0.4],
                  [0.1, 0.3, 1.0, 0.6],
                  [0.2, 0.4, 0.6, 1.0]])
    intra, inter = coact.collaboration(P, np.array([[0, 1], [2, 3]]))
    np.testing.assert_allclose(intra, [0.5, 0.6])
    np.testing.assert_allclose(inter[0, 1], (0.1 + 0.2 + 0.3 + 0.4) / 4)
    np.testing.assert_allclose(inter[1, 0], inter[0, 1])
