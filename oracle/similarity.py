"""Expert similarity table T (oracle), Occult paper App. A.3, Eq. 6-8.

Test infrastructure: only the tests, the smoke check and the benchmark's CPU
baseline use this package; the CUDA library shares no code with it.

T[i, j] is the cosine similarity of columns i and j of the profiled router
logits H [N_ori, Ne] (Eq. 6).  Eq. 7-8 compute its square from inner products
that add up over batches of profiled tokens: the accumulator is the Gram matrix
G = H^T H, summed batch by batch, and T^2[i, j] = G[i, j]^2 / (G[i, i] G[j, j])
(Eq. 8's 1/N_ori factors cancel).  Reading: the table keeps the sign of G[i, j],
    T_signed[i, j] = sign(G[i, j]) * G[i, j]^2 / (G[i, i] * G[j, j]),
which orders experts exactly as the cosine of Eq. 6 does (the square root is
monotone); "most similar" means the largest value.  A column of zeros has
similarity 0 to every expert.
"""
from __future__ import annotations

from typing import Iterable

import numpy as np


def accumulate(G: np.ndarray, logits_batch: np.ndarray) -> np.ndarray:
    """G += H_b^T H_b for one batch of profiled router logits H_b [n, Ne] (fp64)."""
    H = np.asarray(logits_batch, dtype=np.float64)
    G += H.T @ H
    return G


def finish(G: np.ndarray) -> np.ndarray:
    """The signed squared similarity table [Ne, Ne] from the accumulated G (Eq. 8)."""
    G = np.asarray(G, dtype=np.float64)
    diag = np.diag(G)
    den = np.outer(diag, diag)
    out = np.zeros_like(G)
    nz = den > 0
    out[nz] = np.sign(G[nz]) * G[nz] ** 2 / den[nz]
    return out


def table(batches: Iterable[np.ndarray], n_experts: int) -> np.ndarray:
    """Eq. 8 over a sequence of profiled logit batches."""
    G = np.zeros((n_experts, n_experts))
    for b in batches:
        accumulate(G, b)
    return finish(G)
