"""Pins of the oracle's collaboration pruning (Sec. 3.3) against hand-worked
examples, brute force and the invariants the rules imply."""
import numpy as np
import pytest

from oracle import routing


@pytest.fixture
def ex(golden):
    return golden("pruning_worked_example.json")


def test_score_pruned_worked_example(ex):
    e2v = np.array(ex["expert_to_vdev"])
    sp = ex["score_pruned"]
    logits = np.array([c["logits"] for c in sp["cases"]], dtype=np.float32)
    ids, gates, kept = routing.route_score_pruned(logits, sp["top_k"], e2v, sp["n_keep"])
    for t, c in enumerate(sp["cases"]):
        assert kept[t] == c["kept"], c["derivation"]
        assert ids[t].tolist() == c["ids"], c["derivation"]
    # unrenormalised gates are the softmax probabilities exp(z_e) / sum exp(z)
    z = logits.astype(np.float64)
    p = np.exp(z) / np.exp(z).sum(1, keepdims=True)
    np.testing.assert_allclose(gates, np.take_along_axis(p, ids.astype(int), 1), rtol=1e-6)


def test_similarity_pruned_worked_example(ex):
    e2v = np.array(ex["expert_to_vdev"])
    tab = np.array(ex["similarity_pruned"]["table"])
    for c in ex["similarity_pruned"]["cases"]:
        logits = np.array([c["logits"]], dtype=np.float32)
        ids, gates, routed, kept = routing.route_similarity_pruned(
            logits, c["top_k"], e2v, c["n_keep"], tab)
        assert routed[0].tolist() == c["routed"], c["derivation"]
        assert ids[0].tolist() == c["ids"], c["derivation"]
        # the gates stay with the slots: the routed experts' probabilities
        z = logits[0].astype(np.float64)
        p = np.exp(z) / np.exp(z).sum()
        np.testing.assert_allclose(gates[0], p[c["routed"]], rtol=1e-6)


def _random_case(seed, T=200, Ne=16, Nd=4):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, Ne)).astype(np.float32)
    e2v = rng.permutation(np.repeat(np.arange(Nd), Ne // Nd))
    return logits, e2v


@pytest.mark.parametrize("k,n_keep", [(4, 1), (4, 2), (6, 2), (3, 3)])
def test_score_pruned_matches_brute_force(k, n_keep):
    """Brute force over every set of k experts inside the kept devices: the chosen
    set has the largest summed logit (top-k by logit)."""
    logits, e2v = _random_case(k * 10 + n_keep)
    T, Ne = logits.shape
    ids, _, kept = routing.route_score_pruned(logits, k, e2v, n_keep, renorm=True)
    routed, _ = routing.route_topk(logits, k)
    import itertools
    for t in range(T):
        # kept devices: first n_keep distinct devices along the routed experts
        order = []
        for e in routed[t]:
            if e2v[e] not in order:
                order.append(int(e2v[e]))
        assert kept[t] == order[:n_keep]
        allowed = [e for e in range(Ne) if e2v[e] in kept[t]]
        best = max(itertools.combinations(allowed, k),
                   key=lambda s: (sum(float(logits[t, e]) for e in s)))
        assert set(ids[t].tolist()) == set(best)
        assert len(set(ids[t].tolist())) == k


def test_score_pruned_special_cases():
    logits, e2v = _random_case(7)
    k = 4
    # keeping every device is plain top-k
    ids, gates, _ = routing.route_score_pruned(logits, k, e2v, n_keep=4)
    ids0, gates0 = routing.route_topk(logits, k)
    assert (ids == ids0).all()
    np.testing.assert_array_equal(gates, gates0)
    # one kept device: every chosen expert is on the device of the best expert
    ids1, g1, _ = routing.route_score_pruned(logits, k, e2v, n_keep=1, renorm=True)
    assert (e2v[ids1] == e2v[ids0[:, :1]]).all()
    np.testing.assert_allclose(g1.sum(1), 1.0, rtol=1e-12)
    # C_T <= n_keep for every token (n_keep devices hold n_keep * 4 >= k experts)
    for n_keep, kk in ((1, 4), (2, 6), (3, 6)):
        ids2, _, _ = routing.route_score_pruned(logits, kk, e2v, n_keep)
        assert max(len(set(e2v[r].tolist())) for r in ids2) <= n_keep
    with pytest.raises(ValueError):
        routing.route_score_pruned(logits, 6, e2v, 1)


def test_similarity_pruned_invariants():
    logits, e2v = _random_case(11)
    T, Ne = logits.shape
    rng = np.random.default_rng(12)
    tab = rng.standard_normal((Ne, Ne)).astype(np.float32)
    k, n_keep = 6, 2
    ids, gates, routed, kept = routing.route_similarity_pruned(logits, k, e2v, n_keep, tab)
    _, g0 = routing.route_topk(logits, k)
    np.testing.assert_array_equal(gates, g0)
    for t in range(T):
        assert len(set(ids[t].tolist())) == k
        assert set(e2v[ids[t]].tolist()) <= set(kept[t])
        for j in range(k):
            if e2v[routed[t, j]] in kept[t]:
                assert ids[t, j] == routed[t, j]
            else:
                # the replacement is at least as similar as every expert that was
                # still free when slot j was filled
                used = set(ids[t, :j].tolist()) | {int(e) for e in routed[t] if e2v[e] in kept[t]}
                free = [c for c in range(Ne) if e2v[c] in kept[t] and c not in used]
                assert ids[t, j] in free
                assert tab[routed[t, j], ids[t, j]] == max(tab[routed[t, j], c] for c in free)


def test_similarity_pruned_identity_when_nothing_outside():
    logits, e2v = _random_case(13)
    tab = np.zeros((16, 16), dtype=np.float32)
    ids, _, routed, _ = routing.route_similarity_pruned(logits, 4, e2v, 4, tab)
    assert (ids == routed).all()
