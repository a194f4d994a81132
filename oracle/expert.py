"""MoE layer output by its definition (oracle).

Occult paper, Sec. 2.1, Eq. 1: MoE(x) = sum_i R(x)_i * E_i(x).  Without pruning
Occult reaches exactly this result (Sec. 3.2 "maintaining exact computation
results"), so Eq. 1 is the oracle for the layer output.

The pages name the experts' first and second linear layers but no activation;
each expert here is a SwiGLU feed-forward network,
    E(x) = W_d (silu(W_g x) * (W_u x)),
with ``w1[e]`` = [W_g; W_u] (2I rows of length d) and ``w2[e]`` = W_d (d rows of
length I).  Shared experts (always on, no routing) add
    s(x) * [W_d^s (silu(W_g^s x) * (W_u^s x))],
where several shared experts are stacked along the intermediate axis (a sum of
SwiGLU experts equals one SwiGLU expert over the concatenated hidden units) and
s(x) = sigmoid(w_sg . x) when a shared gate is used, else 1.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def swiglu_expert(x: np.ndarray, w1: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """E(x) for the rows of x, fp64.  x [n, d], w1 [2I, d], w2 [d, I] -> [n, d]."""
    x = np.asarray(x, dtype=np.float64)
    w1 = np.asarray(w1, dtype=np.float64)
    w2 = np.asarray(w2, dtype=np.float64)
    I = w1.shape[0] // 2
    g = x @ w1[:I].T
    u = x @ w1[I:].T
    return (silu(g) * u) @ w2.T


def moe_dense(x: np.ndarray, R: np.ndarray, w1: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """Eq. 1 literally: every expert runs on every token and R weights them.

    R [T, Ne] is the router output of Eq. 2 (zero outside the top k).  Costs Ne/k
    times the sparse form; for tiny layers only.
    """
    T, Ne = R.shape
    y = np.zeros((T, x.shape[1]), dtype=np.float64)
    for i in range(Ne):
        y += R[:, i:i + 1] * swiglu_expert(x, w1[i], w2[i])
    return y


def moe_topk(x: np.ndarray, ids: np.ndarray, gates: np.ndarray, w1: np.ndarray,
             w2: np.ndarray, tokens: Optional[Sequence[int]] = None) -> np.ndarray:
    """Eq. 1 summed over the k non-zero router entries only.

    Each expert is evaluated once on the tokens that chose it, then every token
    sums its k gated expert outputs in the order of its ``ids``.  ``tokens``
    restricts the work to a subset of rows (returned in that order).
    """
    if tokens is None:
        tokens = np.arange(ids.shape[0])
    tokens = np.asarray(tokens, dtype=np.int64)
    sub_ids = np.asarray(ids)[tokens]
    sub_g = np.asarray(gates, dtype=np.float64)[tokens]
    xs = np.asarray(x)[tokens]
    n, k = sub_ids.shape
    out = np.zeros((n, k, x.shape[1]), dtype=np.float64)
    for e in np.unique(sub_ids):
        rows, slots = np.nonzero(sub_ids == e)
        out[rows, slots] = swiglu_expert(xs[rows], w1[e], w2[e])
    y = np.zeros((n, x.shape[1]), dtype=np.float64)
    for j in range(k):
        y += sub_g[:, j:j + 1] * out[:, j]
    return y


def shared_gate(x: np.ndarray, w_sg: Optional[np.ndarray]) -> np.ndarray:
    """s(x) = sigmoid(w_sg . x) per row, or ones without a gate vector."""
    x = np.asarray(x, dtype=np.float64)
    if w_sg is None:
        return np.ones(x.shape[0], dtype=np.float64)
    z = x @ np.asarray(w_sg, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-z))


def shared_experts(x: np.ndarray, ws1: np.ndarray, ws2: np.ndarray,
                   w_sg: Optional[np.ndarray] = None,
                   tokens: Optional[Sequence[int]] = None) -> np.ndarray:
    """Always-on shared expert output s(x) * E_shared(x), fp64 [n, d]."""
    if tokens is not None:
        x = np.asarray(x)[np.asarray(tokens, dtype=np.int64)]
    return shared_gate(x, w_sg)[:, None] * swiglu_expert(x, ws1, ws2)


def layer_output(x, ids, gates, weights: dict, tokens=None) -> np.ndarray:
    """Routed experts (Eq. 1) plus the shared experts, if the weights hold any."""
    y = moe_topk(x, ids, gates, weights["w1"], weights["w2"], tokens)
    if "ws1" in weights:
        y = y + shared_experts(x, weights["ws1"], weights["ws2"], weights.get("w_sg"), tokens)
    return y
