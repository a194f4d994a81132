"""Algorithm 1, expert placement rescheduling (oracle).

Occult paper, Sec. 3.2, Algorithm 1 ("Building expert placement"): a greedy,
farthest-point-style partition of the collaboration graph P into Nd equal
device lists.

* Device 0 starts with the two most collaborative experts, i.e. the (i, j),
  i != j, with the largest P[i, j]; equal values go to the first pair in
  row-major order.
* Every later device starts with the unused expert whose mean collaboration
  with all experts placed so far is smallest.
* Each device then repeatedly takes the unused expert whose mean collaboration
  with the experts already on that device is largest, until it holds Ne/Nd
  experts (the printed loop condition "len <= Ne/Nd" would overfill by one;
  it is read as "<").

Readings: the garbled "1/L[d]" is 1/|L[d]|; "|L|" is the number of experts
placed so far.  Both denominators are the same for every candidate, and P is C
scaled by a positive constant, so every comparison is made exactly on integer
sums of C.  Ties go to the lowest expert id.  With Ne/Nd = 1 device 0 keeps only
the first expert of the pair.
"""
from __future__ import annotations

import numpy as np


def place(C: np.ndarray, n_vdev: int) -> np.ndarray:
    """Algorithm 1 on the co-activation counts C [Ne, Ne].  Returns int32 [Nd, Ne/Nd]."""
    C = np.asarray(C, dtype=np.int64)
    Ne = C.shape[0]
    if Ne % n_vdev:
        raise ValueError("Ne must be divisible by Nd")
    n_loc = Ne // n_vdev
    L = [[] for _ in range(n_vdev)]
    used = []
    for d in range(n_vdev):
        if d == 0:
            best = None
            for i in range(Ne):
                for j in range(Ne):
                    if i != j and (best is None or C[i, j] > C[best[0], best[1]]):
                        best = (i, j)
            i, j = best
            L[0].append(i)
            used.append(i)
            if n_loc >= 2:
                L[0].append(j)
                used.append(j)
        else:
            best_e, best_v = None, None
            for e in range(Ne):
                if e in used:
                    continue
                v = sum(int(C[t, e]) for t in used)
                if best_v is None or v < best_v:
                    best_e, best_v = e, v
            L[d].append(best_e)
            used.append(best_e)
        while len(L[d]) < n_loc:
            best_e, best_v = None, None
            for e in range(Ne):
                if e in used:
                    continue
                v = sum(int(C[t, e]) for t in L[d])
                if best_v is None or v > best_v:
                    best_e, best_v = e, v
            L[d].append(best_e)
            used.append(best_e)
    return np.array(L, dtype=np.int32)


def trivial(n_experts: int, n_vdev: int) -> np.ndarray:
    """Contiguous placement: device d holds experts d*n_loc .. (d+1)*n_loc - 1."""
    n_loc = n_experts // n_vdev
    return np.arange(n_experts, dtype=np.int32).reshape(n_vdev, n_loc)


def expert_to_vdev(placement: np.ndarray) -> np.ndarray:
    placement = np.asarray(placement)
    e2v = np.empty(placement.size, dtype=np.int32)
    for d in range(placement.shape[0]):
        for e in placement[d]:
            e2v[int(e)] = d
    return e2v
