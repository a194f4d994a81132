"""Router of the MoE layer (oracle).

Occult paper, Sec. 2.1, Eq. 2: R(x) = Top-K(Softmax(g(x)), k); entries outside the
top k are zero.  The router projection g(.) is not part of this layer's input:
the logits g(x) arrive as an fp32 tensor.

Readings of what Eq. 2 leaves open:

* the top-k set is chosen on the fp32 logits (softmax is monotone, so it is the
  same set) so that the choice does not depend on how exp() rounds; equal logits
  go to the lower expert id; the k ids are listed by descending logit;
* gates are the softmax probabilities of the chosen experts, optionally
  renormalised to sum to one over the k chosen experts.

Device-limited pruning (Sec. 3.3 restricts each token's experts to a few
devices): the devices kept for a token are the ``n_keep`` devices with the
largest summed softmax probability over all of their experts (equal masses go
to the lower device id); top-k is then taken among the experts of the kept
devices, and the gates are renormalised over the k chosen experts.
"""
from __future__ import annotations

import numpy as np


def softmax(logits: np.ndarray) -> np.ndarray:
    """Softmax over the last axis in fp64 (Eq. 2)."""
    z = np.asarray(logits, dtype=np.float64)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def _rank_by_logit(logits: np.ndarray) -> np.ndarray:
    """Expert ids of each row ordered by descending logit, then ascending id."""
    logits = np.asarray(logits, dtype=np.float32)
    T, Ne = logits.shape
    ids = np.broadcast_to(np.arange(Ne), (T, Ne))
    # np.lexsort sorts by the last key first: primary -logit, secondary id
    return np.lexsort((ids, -logits), axis=-1)


def route_topk(logits: np.ndarray, k: int, renorm: bool = False):
    """Top-k softmax routing (Eq. 2).

    Returns ``ids`` int32 [T, k] (descending logit) and ``gates`` fp64 [T, k].
    """
    p = softmax(logits)
    order = _rank_by_logit(logits)[:, :k]
    gates = np.take_along_axis(p, order, axis=-1)
    if renorm:
        gates = gates / gates.sum(axis=-1, keepdims=True)
    return order.astype(np.int32), gates


def gate_matrix(ids: np.ndarray, gates: np.ndarray, n_experts: int) -> np.ndarray:
    """The dense R(x) of Eq. 2: [T, Ne] with the gates at the chosen ids, else 0."""
    T = ids.shape[0]
    R = np.zeros((T, n_experts), dtype=np.float64)
    for t in range(T):
        for j in range(ids.shape[1]):
            R[t, ids[t, j]] = gates[t, j]
    return R


def device_mass(logits: np.ndarray, expert_to_vdev: np.ndarray, n_vdev: int) -> np.ndarray:
    """Summed softmax probability of every device's experts, fp64 [T, Nd]."""
    p = softmax(logits)
    mass = np.zeros((p.shape[0], n_vdev), dtype=np.float64)
    for e, d in enumerate(np.asarray(expert_to_vdev)):
        mass[:, d] += p[:, e]
    return mass


def route_device_limited(logits: np.ndarray, k: int, expert_to_vdev: np.ndarray,
                         n_vdev: int, n_keep: int):
    """Device-limited pruning: keep ``n_keep`` devices by summed gate mass, then top-k.

    Returns ``ids`` int32 [T, k], renormalised ``gates`` fp64 [T, k], the kept
    devices int32 [T, n_keep] (descending mass) and the relative mass margin
    between the last kept and the first dropped device (``inf`` when none is
    dropped).  A margin near zero means the choice hangs on rounding.
    """
    logits = np.asarray(logits, dtype=np.float32)
    e2v = np.asarray(expert_to_vdev)
    T, Ne = logits.shape
    p = softmax(logits)
    mass = device_mass(logits, e2v, n_vdev)
    dev_ids = np.broadcast_to(np.arange(n_vdev), (T, n_vdev))
    dev_order = np.lexsort((dev_ids, -mass), axis=-1)
    kept = dev_order[:, :n_keep]
    if n_keep < n_vdev:
        m_last = np.take_along_axis(mass, kept[:, -1:], axis=-1)[:, 0]
        m_next = np.take_along_axis(mass, dev_order[:, n_keep:n_keep + 1], axis=-1)[:, 0]
        margin = (m_last - m_next) / m_last
    else:
        margin = np.full(T, np.inf)
    ids = np.empty((T, k), dtype=np.int32)
    gates = np.empty((T, k), dtype=np.float64)
    ranked = _rank_by_logit(logits)
    for t in range(T):
        allowed = set(int(d) for d in kept[t])
        chosen = [int(e) for e in ranked[t] if int(e2v[e]) in allowed][:k]
        ids[t] = chosen
        g = p[t, chosen]
        gates[t] = g / g.sum()
    return ids, gates, kept.astype(np.int32), margin


def token_devices(ids: np.ndarray, expert_to_vdev: np.ndarray, n_vdev: int) -> np.ndarray:
    """Boolean [T, Nd]: token t activates at least one expert kept on device d."""
    e2v = np.asarray(expert_to_vdev)
    T = ids.shape[0]
    act = np.zeros((T, n_vdev), dtype=bool)
    for t in range(T):
        for e in ids[t]:
            act[t, e2v[e]] = True
    return act
