"""Pins of the sharded-source exchange plan (oracle)."""
import numpy as np

from oracle import brim as obrim
from oracle import shard


def test_worked_example(golden):
    g = golden("shard_worked_example.json")
    b0s, counts, send_off, recv_off = shard.shard_plan(np.array(g["act"], bool), g["src_off"])
    assert b0s.tolist() == g["brim0_send"], g["derivation"]
    assert counts.tolist() == g["counts"]
    assert send_off.tolist() == g["send_off"]
    assert recv_off.tolist() == g["recv_off"]


def _random(seed, T=300, Nd=8, n_src=5):
    rng = np.random.default_rng(seed)
    act = rng.random((T, Nd)) < 0.35
    cuts = np.sort(rng.choice(np.arange(1, T), n_src - 1, replace=False))
    return act, [0, *cuts.tolist(), T]


def test_exchange_reaches_the_single_source_layout():
    """Dispatch per source, then the exchange, gives the single-source SFD tensor;
    the reverse exchange brings it back; every row is moved exactly once."""
    act, src_off = _random(0)
    T, Nd = act.shape
    x = np.random.default_rng(1).standard_normal((T, 6))
    b0 = obrim.build_brim0(act)
    b0s, counts, send_off, recv_off = shard.shard_plan(act, src_off)
    n_sfd = int(act.sum())
    assert counts.sum() == n_sfd
    # the send map is a bijection onto [0, N_sfd)
    assert sorted(b0s[b0s >= 0].tolist()) == list(range(n_sfd))
    x_send = obrim.dispatch(x, b0s)
    x_recv = shard.all_to_all(x_send, counts, send_off, recv_off)
    np.testing.assert_array_equal(x_recv, obrim.dispatch(x, b0))
    np.testing.assert_array_equal(shard.all_to_all(x_recv, counts, send_off, recv_off,
                                                   reverse=True), x_send)
    # element by element: (d, t) lands where single-source BRIM0 puts it
    for s in range(len(src_off) - 1):
        for d in range(Nd):
            toks = [t for t in range(src_off[s], src_off[s + 1]) if act[t, d]]
            assert [int(b0s[d, t]) for t in toks] == list(range(send_off[s, d],
                                                                send_off[s, d] + len(toks)))
            assert [int(b0[d, t]) for t in toks] == list(range(recv_off[s, d],
                                                               recv_off[s, d] + len(toks)))


def test_special_cases():
    act, _ = _random(2, T=64)
    b0 = obrim.build_brim0(act)
    # one source: the send layout is the single-source layout
    b0s, counts, send_off, recv_off = shard.shard_plan(act, [0, 64])
    np.testing.assert_array_equal(b0s, b0)
    np.testing.assert_array_equal(send_off, recv_off)
    # empty shards move nothing
    b0s, counts, _, _ = shard.shard_plan(act, [0, 0, 30, 30, 64])
    assert not counts[0].any() and not counts[2].any()
    np.testing.assert_array_equal(b0s >= 0, b0 >= 0)
