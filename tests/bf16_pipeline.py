"""CPU emulation of the rounding the bf16 GPU path performs in the expert FFN,
forward and backward (test infrastructure: it checks that the per-element error
bounds of ``layer_cases`` are neither violated nor vacuous).

It follows the GPU's precision choices, not its kernels: every contraction takes
bf16 operands and accumulates in fp32 (here an fp32 BLAS product, whose order of
additions differs from the tensor cores' but obeys the same fp32 accumulation
bound), elementwise work is fp32, and values are rounded to bf16 exactly where
the GPU stores bf16:
  forward   G = a W_g^T, U = a W_u^T (fp32); h' = g silu(G) U rounded to bf16;
            y_epd = h' W_d^T (fp32); a token's rows summed in fp32;
  backward  G, U as saved by the forward (bf16); dh' = dy W_d (fp32);
            dg = <dh', silu(G) U> (fp32); dG, dU rounded to bf16;
            dx rows = [dG | dU] [W_g; W_u] (fp32); dW_d = dy^T h'; dW_g|u = [dG|dU]^T a.

``mistake`` plants one error of the kind a kernel bug makes, for the tests that
show a bound catches it:
  "drop_row"        the first row contributes nothing (h' row zero, no dW terms);
  "gate_twice"      the routing weight multiplies twice;
  "neighbour"       the weights of expert e + 1 (mod Ne) are used.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch


def bf16(a) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even), returned as fp32."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def mm32(a, b) -> np.ndarray:
    """fp32 product of two fp32 matrices (fp32 accumulation)."""
    return np.asarray(a, dtype=np.float32) @ np.asarray(b, dtype=np.float32)


def _sigmoid32(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.float32)
    return (np.float32(1.0) / (np.float32(1.0) + np.exp(-z))).astype(np.float32)


def _weights(w1, w2, e: int, mistake: Optional[str]):
    if mistake == "neighbour":
        e = (e + 1) % w1.shape[0]
    I = w1.shape[1] // 2
    return w1[e, :I], w1[e, I:], w2[e]


def forward_rows(a, w1, w2, e: int, gate, mistake: Optional[str] = None):
    """One expert's EPD rows (a [n, d] token inputs, gate [n]): G, U (fp32), h'
    (bf16 values) and y_epd (fp32)."""
    wg, wu, wd = _weights(w1, w2, e, mistake)
    g = np.asarray(gate, dtype=np.float32)[:, None]
    if mistake == "gate_twice":
        g = g * g
    G = mm32(a, wg.T)
    U = mm32(a, wu.T)
    h = bf16(g * (G * _sigmoid32(G)) * U)
    if mistake == "drop_row" and len(h):
        h[0] = 0.0
    return {"G": G, "U": U, "h": h, "y_epd": mm32(h, wd.T)}


def backward_rows(a, dy, w1, w2, e: int, gate, fwd, mistake: Optional[str] = None):
    """One expert's rows of the backward, from the forward's saved values ``fwd``:
    dg [n], dx rows [n, d] (fp32), dW1 [2I, d] and dW2 [d, I] (fp32)."""
    wg, wu, wd = _weights(w1, w2, e, mistake)
    g = np.asarray(gate, dtype=np.float32)[:, None]
    if mistake == "gate_twice":
        g = g * g
    Gs, Us = bf16(fwd["G"]), bf16(fwd["U"])
    dhp = mm32(dy, wd)
    sig = _sigmoid32(Gs)
    s = Gs * sig
    dg = np.sum(dhp * (s * Us), axis=1, dtype=np.float32)
    dh = g * dhp
    dG = bf16(dh * Us * sig * (np.float32(1.0) + Gs * (np.float32(1.0) - sig)))
    dU = bf16(dh * s)
    h = fwd["h"]
    if mistake == "drop_row" and len(h):
        dG, dU, h, dy = dG.copy(), dU.copy(), h.copy(), dy.copy()
        dG[0] = dU[0] = 0.0
        dy[0] = 0.0
    dgu = np.concatenate([dG, dU], axis=1)
    dx = mm32(dgu, np.concatenate([wg, wu], axis=0))
    dW1 = np.concatenate([mm32(dG.T, a), mm32(dU.T, a)], axis=0)
    dW2 = mm32(dy.T, h)
    return {"dg": dg, "dx_rows": dx, "dW1": dW1, "dW2": dW2}
