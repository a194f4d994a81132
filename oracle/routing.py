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

Collaboration pruning as Sec. 3.3 itself states it: the kept devices are found
by walking the token's k routed experts in descending routing score and
collecting their devices until ``n_keep`` are reached (all of them when the k
experts cover fewer).  Then either
* routing-score-based pruning: all Ne scores are sorted in descending order and
  the top k experts lying on the kept devices are selected, or
* expert-similarity-based pruning: the k routed experts are walked in
  descending score; an expert on a kept device stays, one outside is replaced
  by the most similar expert of the table T (App. A.3) that lies on a kept
  device and is not selected yet.
Readings where Sec. 3.3 is silent: scores are compared on the fp32 logits with
ties to the lower id, as for top-k; the gates of score-based pruning are the
softmax probabilities of the selected experts (renormalised over them when
``renorm``); in similarity-based pruning the experts kept in place are counted
as selected before any replacement is made, a replacement takes over the
replaced slot and its routing weight, similarities are compared as fp32 with
ties to the lower id, and the slots keep the routed experts' descending-score
order.
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


def _check_pruning(expert_to_vdev, k: int, n_keep: int) -> None:
    """Every expert set inside n_keep devices must be able to hold k experts."""
    counts = np.bincount(np.asarray(expert_to_vdev))
    if n_keep < 1 or np.sort(counts)[:n_keep].sum() < k:
        raise ValueError("pruning needs n_keep devices that hold at least k experts")


def pruning_devices(ids: np.ndarray, expert_to_vdev: np.ndarray, n_keep: int) -> list:
    """Sec. 3.3: per token, the devices of its routed experts (``ids`` in descending
    score) in order of first appearance, stopping once ``n_keep`` are collected."""
    e2v = np.asarray(expert_to_vdev)
    out = []
    for row in np.asarray(ids):
        kept = []
        for e in row:
            d = int(e2v[int(e)])
            if d not in kept:
                if len(kept) == n_keep:
                    break
                kept.append(d)
        out.append(kept)
    return out


def route_score_pruned(logits: np.ndarray, k: int, expert_to_vdev: np.ndarray, n_keep: int,
                       renorm: bool = False):
    """Routing-score-based pruning (Sec. 3.3, steps 1-2).

    Returns ``ids`` int32 [T, k] (descending logit), ``gates`` fp64 [T, k] and the
    kept devices of every token (a list of lists, order of first appearance).
    """
    _check_pruning(expert_to_vdev, k, n_keep)
    logits = np.asarray(logits, dtype=np.float32)
    e2v = np.asarray(expert_to_vdev)
    T = logits.shape[0]
    routed, _ = route_topk(logits, k)
    kept = pruning_devices(routed, e2v, n_keep)
    p = softmax(logits)
    ranked = _rank_by_logit(logits)          # step 1: all scores, descending
    ids = np.empty((T, k), dtype=np.int32)
    gates = np.empty((T, k), dtype=np.float64)
    for t in range(T):
        allowed = set(kept[t])
        chosen = [int(e) for e in ranked[t] if int(e2v[e]) in allowed][:k]   # step 2
        ids[t] = chosen
        g = p[t, chosen]
        gates[t] = g / g.sum() if renorm else g
    return ids, gates, kept


def route_similarity_pruned(logits: np.ndarray, k: int, expert_to_vdev: np.ndarray,
                            n_keep: int, table: np.ndarray, renorm: bool = False):
    """Expert-similarity-based pruning (Sec. 3.3) with similarity table ``table``
    [Ne, Ne] (row e: similarity of expert e to every expert).

    Returns ``ids`` int32 [T, k] (slot j holds routed expert j or its
    replacement), ``gates`` fp64 [T, k] (the routed experts' weights, top-k
    softmax probabilities renormalised when ``renorm``), ``routed`` int32 [T, k]
    (the experts whose probabilities the gates are) and the kept devices.
    """
    _check_pruning(expert_to_vdev, k, n_keep)
    logits = np.asarray(logits, dtype=np.float32)
    e2v = np.asarray(expert_to_vdev)
    tab = np.asarray(table, dtype=np.float32)
    T, Ne = logits.shape
    routed, gates = route_topk(logits, k, renorm=renorm)
    kept = pruning_devices(routed, e2v, n_keep)
    ids = routed.copy()
    for t in range(T):
        allowed = set(kept[t])
        selected = set(int(e) for e in routed[t] if int(e2v[e]) in allowed)
        for j, e in enumerate(routed[t]):
            e = int(e)
            if int(e2v[e]) in allowed:
                continue
            best = None
            for c in range(Ne):                  # ascending id: ties keep the lower id
                if int(e2v[c]) not in allowed or c in selected:
                    continue
                if best is None or tab[e, c] > tab[e, best]:
                    best = c
            selected.add(best)
            ids[t, j] = best
    return ids, gates, routed, kept
