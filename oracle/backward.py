"""Gradients of the MoE layer output (oracle), fp64.

Occult paper, Sec. 1: the sparse kernels serve the forward and the backward
pass; the pages give no backward pseudo-code.  The backward of Eq. 1,
    y_t = sum_j g_tj * W_d[e] (silu(W_g[e] x_t) * (W_u[e] x_t)),   e = e_tj,
is its plain derivative.  With G = W_g x, U = W_u x, s = silu(G), h = s * U
and an upstream gradient dy_t:
    dW_d[e] += g dy_t h^T                    dg_tj = <dy_t, W_d[e] h>
    dh       = g W_d[e]^T dy_t               dG = dh * U * silu'(G),  dU = dh * s
    dW_g[e] += dG x_t^T,  dW_u[e] += dU x_t^T
    dx_t    += W_g[e]^T dG + W_u[e]^T dU
with silu'(G) = sigma(G) (1 + G (1 - sigma(G))).  moe_backward takes the gates as
given; router_grad carries dgates on into the router logits through the softmax
of Eq. 2.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import numpy as np

from .routing import softmax


def _sigmoid(z: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-z))


def moe_backward(x: np.ndarray, ids: np.ndarray, gates: np.ndarray, w1: np.ndarray,
                 w2: np.ndarray, dy: np.ndarray,
                 experts: Optional[Sequence[int]] = None) -> Dict[str, np.ndarray]:
    """dx [T, d], dw1 [Ne, 2I, d], dw2 [Ne, d, I], dgates [T, k] of sum_t <dy_t, y_t>.

    ``experts`` restricts the computation to those experts: the other experts'
    weight gradients stay zero, and dx / dgates hold only the listed experts'
    contributions (the full gradients are the sums over disjoint expert sets).
    """
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    ids = np.asarray(ids)
    gates = np.asarray(gates, dtype=np.float64)
    Ne, two_i, d = w1.shape
    I = two_i // 2
    T, k = ids.shape
    dx = np.zeros((T, d))
    dw1 = np.zeros((Ne, two_i, d))
    dw2 = np.zeros((Ne, d, I))
    dgates = np.zeros((T, k))
    todo = np.unique(ids) if experts is None else [int(e) for e in experts]
    for e in todo:
        rows, slots = np.nonzero(ids == e)
        wg = np.asarray(w1[e, :I], dtype=np.float64)
        wu = np.asarray(w1[e, I:], dtype=np.float64)
        wd = np.asarray(w2[e], dtype=np.float64)
        a = x[rows]                          # [n, d]
        g = gates[rows, slots][:, None]      # [n, 1]
        G = a @ wg.T
        U = a @ wu.T
        sig = _sigmoid(G)
        s = G * sig
        h = s * U
        dyr = dy[rows]                       # [n, d]
        dhp = dyr @ wd                       # gradient of h' = g h, [n, I]
        dgates[rows, slots] = np.sum(dhp * h, axis=1)
        dh = g * dhp
        dG = dh * U * sig * (1.0 + G * (1.0 - sig))
        dU = dh * s
        dx[rows] += dG @ wg + dU @ wu        # a token holds an expert at most once
        dw2[e] = dyr.T @ (g * h)
        dw1[e, :I] = dG.T @ a
        dw1[e, I:] = dU.T @ a
    return {"dx": dx, "dw1": dw1, "dw2": dw2, "dgates": dgates}


def router_grad(logits: np.ndarray, gate_ids: np.ndarray, dgates: np.ndarray,
                renorm: bool = False) -> np.ndarray:
    """Gradient of sum_tj dgates_tj * g_tj with respect to the router logits z.

    The gates are g_tj = p_t[gate_ids_tj] with p_t = softmax(z_t) (Eq. 2), divided
    by their sum over j when ``renorm``.  The selection of experts is piecewise
    constant in z, so no gradient flows through it.  With q_j = p[e_j] and
    S = sum_j q_j:
        plain:   dz_i = p_i * (sum_j [e_j = i] dg_j - sum_j dg_j g_j)
        renorm:  dz_i = sum_j [e_j = i] g_j * (dg_j - sum_m dg_m g_m),
    (in the renormalised case the logits of unselected experts get no gradient).
    Returns dz fp64 [T, Ne].
    """
    z = np.asarray(logits, dtype=np.float64)
    ids = np.asarray(gate_ids)
    dg = np.asarray(dgates, dtype=np.float64)
    p = softmax(z)
    T, Ne = z.shape
    dz = np.zeros((T, Ne))
    for t in range(T):
        q = p[t, ids[t]]
        g = q / q.sum() if renorm else q
        inner = float(np.dot(dg[t], g))
        if renorm:
            for j, e in enumerate(ids[t]):
                dz[t, e] += g[j] * (dg[t, j] - inner)
        else:
            sel = np.zeros(Ne)
            for j, e in enumerate(ids[t]):
                sel[e] += dg[t, j]
            dz[t] = p[t] * (sel - inner)
    return dz
