"""Pins of the oracle Algorithm 1 (expert placement)."""
import numpy as np
import pytest

import synth
from oracle import coact, placement, routing


def test_worked_example(golden):
    g = golden("placement_worked_example.json")
    L = placement.place(np.array(g["C"]), g["n_vdev"])
    assert L.tolist() == g["expect"]["placement"]


@pytest.mark.parametrize("seed,Ne,Nd", [(0, 16, 4), (1, 12, 3), (2, 32, 8)])
def test_recovers_planted_blocks(seed, Ne, Nd):
    rng = np.random.default_rng(seed)
    n_loc = Ne // Nd
    perm = rng.permutation(Ne)
    block = np.empty(Ne, dtype=int)
    block[perm] = np.repeat(np.arange(Nd), n_loc)
    C = np.zeros((Ne, Ne), dtype=np.int64)
    for i in range(Ne):
        for j in range(Ne):
            if block[i] == block[j]:
                C[i, j] = rng.integers(5, 50) if i != j else 100
    C = np.maximum(C, C.T)
    L = placement.place(C, Nd)
    got = sorted(sorted(r) for r in L.tolist())
    want = sorted(sorted(np.nonzero(block == b)[0].tolist()) for b in range(Nd))
    assert got == want


@pytest.mark.parametrize("seed,Ne,Nd", [(3, 8, 2), (4, 64, 8), (5, 60, 4), (6, 6, 6)])
def test_output_is_equal_partition(seed, Ne, Nd):
    rng = np.random.default_rng(seed)
    C = rng.integers(0, 30, size=(Ne, Ne))
    C = C + C.T
    L = placement.place(C, Nd)
    assert L.shape == (Nd, Ne // Nd)
    assert sorted(L.ravel().tolist()) == list(range(Ne))


def test_rescheduling_lowers_ct_on_clustered_routing():
    """Sec. 3.2 / Table 1: Alg. 1 lowers E[C_T] against the contiguous placement."""
    cfg = synth.CONFIGS["olmoe_fwd"]
    prof = synth.profiling_logits(cfg).numpy()[:4096]
    ids_p, _ = routing.route_topk(prof, cfg.top_k)
    L = placement.place(coact.coactivation(ids_p, cfg.n_experts), cfg.n_vdev)
    ids, _ = routing.route_topk(synth.measured_logits(cfg, 2048).numpy(), cfg.top_k)
    ct_alg1 = coact.replicas_per_token(ids, placement.expert_to_vdev(L)).mean()
    ct_triv = coact.replicas_per_token(
        ids, placement.expert_to_vdev(placement.trivial(cfg.n_experts, cfg.n_vdev))).mean()
    assert ct_alg1 < ct_triv
