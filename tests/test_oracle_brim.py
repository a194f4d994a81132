"""Pins of the oracle BRIMs (Alg. 3, 5), dispatch/combine (Alg. 4, 9) and the
staged pipeline (Alg. 2) against hand-worked values, invariants and Eq. 1."""
import numpy as np
import pytest

from oracle import brim, coact, expert, placement, routing


def _random_layer(seed, T, Ne, Nd, k, d=8, I=6):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, Ne)).astype(np.float32)
    ids, gates = routing.route_topk(logits, k)
    L = rng.permutation(Ne).reshape(Nd, Ne // Nd).astype(np.int32)
    x = rng.standard_normal((T, d))
    w1 = rng.standard_normal((Ne, 2 * I, d)) * 0.3
    w2 = rng.standard_normal((Ne, d, I)) * 0.3
    return ids, gates, L, x, w1, w2


def test_worked_example(golden):
    g = golden("brim_worked_example.json")
    e = g["expect"]
    b = brim.Brims(np.array(g["ids"]), np.array(g["gates"]), np.array(g["placement"]))
    assert b.brim0.tolist() == e["brim0"]
    assert b.seg_off.tolist() == e["seg_off"]
    assert b.n_sfd == e["n_sfd"]
    assert b.ct.tolist() == e["ct"]
    assert [m.tolist() for m in b.brim1] == e["brim1"]
    assert b.epd_base.tolist() == e["epd_base"]
    assert b.exp_off.tolist() == e["exp_off"]
    assert b.epd_src.tolist() == e["epd_src"]
    assert b.epd_tok.tolist() == e["epd_tok"]
    assert b.epd_exp.tolist() == e["epd_exp"]
    np.testing.assert_allclose(b.epd_gate, e["epd_gate"], rtol=0)


@pytest.mark.parametrize("seed,T,Ne,Nd,k", [(0, 37, 8, 4, 2), (1, 64, 12, 3, 5),
                                            (2, 50, 16, 8, 4), (3, 20, 6, 1, 3),
                                            (4, 33, 8, 8, 8)])
def test_invariants(seed, T, Ne, Nd, k):
    ids, gates, L, *_ = _random_layer(seed, T, Ne, Nd, k)
    b = brim.Brims(ids, gates, L)
    # BRIM0's non-negative entries are a bijection onto [0, N_sfd)
    v = b.brim0[b.brim0 >= 0]
    assert sorted(v.tolist()) == list(range(b.n_sfd))
    # device-major numbering: every entry of device d precedes those of d+1
    for d in range(Nd):
        seg = b.brim0[d][b.brim0[d] >= 0]
        assert (np.diff(seg) == 1).all() if seg.size else True
        assert seg.size == 0 or seg[0] == b.seg_off[d]
    # N_sfd = sum of per-token replica counts, and Eq. 5 bounds every token
    e2v = placement.expert_to_vdev(L)
    ct = coact.replicas_per_token(ids, e2v)
    assert b.n_sfd == ct.sum() == b.ct.sum()
    lo, hi = coact.ct_bounds(k, Ne, Nd)
    assert (ct >= lo).all() and (ct <= hi).all()
    # BRIM1 over all devices is a bijection onto the T*k EPD rows
    assert b.n_epd == T * k
    got = np.concatenate([b.epd_base[d] + m[m >= 0] for d, m in enumerate(b.brim1)])
    assert sorted(got.tolist()) == list(range(T * k))
    # tensor states: ORI <= SFD <= EPD
    assert T <= b.n_sfd <= b.n_epd
    # each EPD row pairs a token with one of its experts, each pair exactly once
    pairs = sorted(zip(b.epd_tok.tolist(), b.epd_exp.tolist()))
    assert pairs == sorted((t, int(e)) for t in range(T) for e in ids[t])
    # the SFD row feeding an EPD row lies on the expert's device and holds its token
    for r in range(b.n_epd):
        dv = e2v[b.epd_exp[r]]
        assert b.seg_off[dv] <= b.epd_src[r] < b.seg_off[dv + 1]
        assert b.brim0[dv, b.epd_tok[r]] == b.epd_src[r]
    # expert segments are contiguous, in placement-slot order
    for s in range(Ne):
        e = L[s // (Ne // Nd), s % (Ne // Nd)]
        seg = b.epd_exp[b.exp_off[s]:b.exp_off[s + 1]]
        assert (seg == e).all()
        assert (np.diff(b.epd_tok[b.exp_off[s]:b.exp_off[s + 1]]) > 0).all()


def test_single_device_reduces_to_plain_expert_sort():
    ids, gates, _, *_ = _random_layer(7, 40, 8, 1, 3)
    L = np.arange(8, dtype=np.int32).reshape(1, 8)
    b = brim.Brims(ids, gates, L)
    assert b.brim0.tolist() == [list(range(40))]
    # EPD order = stable sort of (token, expert) pairs by expert
    order = sorted(((int(e), t) for t in range(40) for e in ids[t]))
    assert list(zip(b.epd_exp.tolist(), b.epd_tok.tolist())) == order


def test_round_trip_identity_experts_gives_k_times_x():
    """Scatter ORI->SFD->EPD then merge EPD->SFD->ORI with identity experts and unit gates."""
    T, Ne, Nd, k, D = 45, 12, 4, 3, 5
    ids, gates, L, *_ = _random_layer(8, T, Ne, Nd, k)
    b = brim.Brims(ids, gates, L)
    x = np.random.default_rng(9).integers(-50, 50, size=(T, D)).astype(np.float32)
    x_sfd = brim.dispatch(x, b.brim0)
    x_epd = np.zeros((b.n_epd, D), np.float32)
    y_sfd = np.zeros((b.n_sfd, D), np.float32)
    for d in range(Nd):
        for j in range(Ne // Nd):
            for r in range(b.brim1[d].shape[1]):
                v = b.brim1[d][j, r]
                if v >= 0:
                    x_epd[b.epd_base[d] + v] = x_sfd[b.seg_off[d] + r]
    for d in range(Nd):
        for j in range(Ne // Nd):
            for r in range(b.brim1[d].shape[1]):
                v = b.brim1[d][j, r]
                if v >= 0:
                    y_sfd[b.seg_off[d] + r] += x_epd[b.epd_base[d] + v]
    y = np.zeros((T, D), np.float32)
    for d in range(Nd):
        for t in range(T):
            if b.brim0[d, t] >= 0:
                y[t] += y_sfd[b.brim0[d, t]]
    np.testing.assert_array_equal(y, k * x)


@pytest.mark.parametrize("seed,T,Ne,Nd,k", [(10, 30, 8, 4, 2), (11, 25, 12, 4, 4),
                                            (12, 16, 6, 3, 6)])
def test_staged_pipeline_equals_eq1(seed, T, Ne, Nd, k):
    """Occult without pruning reaches the standard top-k MoE output (Sec. 3.2)."""
    ids, gates, L, x, w1, w2 = _random_layer(seed, T, Ne, Nd, k)
    y_staged, _ = brim.occult_forward_staged(x, ids, gates, L, w1, w2)
    y_topk = expert.moe_topk(x, ids, gates, w1, w2)
    y_dense = expert.moe_dense(x, routing.gate_matrix(ids, gates, Ne), w1, w2)
    np.testing.assert_allclose(y_staged, y_topk, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(y_dense, y_topk, rtol=1e-12, atol=1e-13)


def test_placement_does_not_change_the_output():
    ids, gates, L, x, w1, w2 = _random_layer(13, 40, 8, 4, 3)
    y_a, st_a = brim.occult_forward_staged(x, ids, gates, L, w1, w2)
    y_b, st_b = brim.occult_forward_staged(x, ids, gates, placement.trivial(8, 4), w1, w2)
    np.testing.assert_allclose(y_a, y_b, rtol=1e-12, atol=1e-13)
    # the EPD tensors hold the same rows, permuted
    np.testing.assert_allclose(np.sort(st_a["h_epd"], axis=0), np.sort(st_b["h_epd"], axis=0),
                               rtol=1e-12, atol=1e-13)


def test_fig2_ct(golden):
    g = golden("fig2_ct_example.json")
    e2v = placement.expert_to_vdev(np.array(g["placement"]))
    ct_b = coact.replicas_per_token(np.array(g["ids_b"]), e2v).mean()
    ct_c = coact.replicas_per_token(np.array(g["ids_c"]), e2v).mean()
    assert g["top_k"] == g["expect"]["ct_conventional"]  # k replicas per token
    assert ct_b == g["expect"]["ct_b"]
    assert ct_c == g["expect"]["ct_c"]
    assert coact.ct_bounds(2, 4, 2) == (g["expect"]["ct_lower_bound"], g["expect"]["ct_upper_bound"])
