"""Co-activation profiling and the communication budget C_T (oracle).

Occult paper:
* Sec. 2.1, Eq. 3: C[i, j] = number of tokens of the batch whose router output
  is non-zero for both expert i and expert j.  As written the formula counts
  i = j too, so the diagonal holds each expert's load.
* Sec. 2.1, Eq. 4: P = C / max_{i,j} C[i, j] (the max runs over all entries,
  the diagonal included).
* Sec. 1 and Sec. 2.2: C_T is the average number of replicas per token, one per
  device holding any of the token's experts; Eq. 5 bounds it by
  ceil(k * Nd / Ne) from below and min(k, Nd) from above.
* Sec. 3.2: intra-collaboration of device d is the mean P over ordered pairs of
  distinct experts on d; inter-collaboration of devices d1, d2 is the mean P
  over expert pairs across them.
"""
from __future__ import annotations

import math

import numpy as np


def coactivation(ids: np.ndarray, n_experts: int) -> np.ndarray:
    """Eq. 3 by brute force over tokens and expert pairs.  int64 [Ne, Ne]."""
    C = np.zeros((n_experts, n_experts), dtype=np.int64)
    for row in np.asarray(ids):
        active = sorted(set(int(e) for e in row))
        for i in active:
            for j in active:
                C[i, j] += 1
    return C


def normalise(C: np.ndarray) -> np.ndarray:
    """Eq. 4: P = C / max C, fp64."""
    m = int(np.max(C))
    return np.asarray(C, dtype=np.float64) / (m if m > 0 else 1)


def replicas_per_token(ids: np.ndarray, expert_to_vdev: np.ndarray) -> np.ndarray:
    """C_T of every token: the number of distinct devices among its experts."""
    e2v = np.asarray(expert_to_vdev)
    return np.array([len(set(int(e2v[e]) for e in row)) for row in np.asarray(ids)],
                    dtype=np.int64)


def ct_histogram(ct: np.ndarray, max_ct: int) -> np.ndarray:
    """Count of tokens with C_T = 0, 1, ..., max_ct.  int64 [max_ct + 1]."""
    h = np.zeros(max_ct + 1, dtype=np.int64)
    for c in np.asarray(ct):
        h[int(c)] += 1
    return h


def ct_bounds(k: int, n_experts: int, n_vdev: int):
    """Eq. 5: (ceil(k * Nd / Ne), min(k, Nd))."""
    return math.ceil(k * n_vdev / n_experts), min(k, n_vdev)


def collaboration(P: np.ndarray, placement: np.ndarray):
    """Sec. 3.2 metrics: C_intra [Nd] and C_inter [Nd, Nd] (diagonal unused)."""
    placement = np.asarray(placement)
    Nd = placement.shape[0]
    intra = np.zeros(Nd, dtype=np.float64)
    inter = np.zeros((Nd, Nd), dtype=np.float64)
    for d in range(Nd):
        L = [int(e) for e in placement[d]]
        pairs = [(i, j) for i in L for j in L if i != j]
        intra[d] = sum(P[i, j] for i, j in pairs) / len(pairs) if pairs else 0.0
        for d2 in range(Nd):
            if d2 == d:
                continue
            L2 = [int(e) for e in placement[d2]]
            inter[d, d2] = sum(P[i, j] for i in L for j in L2) / (len(L) * len(L2))
    return intra, inter
