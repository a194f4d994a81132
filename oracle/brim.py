"""Bidirectional Re-Index Matrices and the staged Occult pipeline (oracle).

Occult paper, Sec. 3.1 (tensor states ORI < SFD < EPD, BRIM) and Appendix A.2
(Algorithms 3-9), written as plain loops.

Single-source reading: one GPU holds the whole batch, so BRIM0 is built once
over all N_ori tokens exactly as Algorithm 3 states, and the first all-to-all
hands device d the SFD rows whose BRIM0[d, *] entry is non-negative, in index
order.  Device d's received SFD rows are therefore the contiguous range
[seg_off[d], seg_off[d+1]) of the dispatched tensor.

EPD layout: Algorithm 5 numbers device d's EPD rows from 0; this build lays the
devices' EPD tensors out one after the other, so the global EPD row of a BRIM1
entry v on device d is epd_base[d] + v, epd_base[d] being the EPD row count of
devices 0..d-1.
"""
from __future__ import annotations

from typing import List, Tuple

import numpy as np


def build_brim0(act: np.ndarray) -> np.ndarray:
    """Algorithm 3.  ``act`` [T, Nd] marks "token t activates an expert on device d".

    BRIM0[d, t] is a running counter taken device by device, token by token, over
    the (d, t) pairs that are active, and -1 elsewhere.  Returns int64 [Nd, T].
    """
    T, Nd = act.shape
    brim0 = np.empty((Nd, T), dtype=np.int64)
    ctr = 0
    for d in range(Nd):
        for t in range(T):
            if act[t, d]:
                brim0[d, t] = ctr
                ctr += 1
            else:
                brim0[d, t] = -1
    return brim0


def segments(brim0: np.ndarray) -> Tuple[np.ndarray, List[np.ndarray]]:
    """Receive segments of the first all-to-all.

    Returns ``seg_off`` [Nd+1] (start of each device's SFD rows) and, for each
    device, the ORI token of each of its SFD rows in row order.
    """
    Nd, T = brim0.shape
    seg_off = np.zeros(Nd + 1, dtype=np.int64)
    rows = []
    for d in range(Nd):
        toks = [t for t in range(T) if brim0[d, t] >= 0]
        toks.sort(key=lambda t: brim0[d, t])
        rows.append(np.array(toks, dtype=np.int64))
        seg_off[d + 1] = seg_off[d] + len(toks)
    return seg_off, rows


def dispatch(x: np.ndarray, brim0: np.ndarray) -> np.ndarray:
    """Algorithm 4: x_sfd[BRIM0[d, t]] = x[t] for every non-negative entry."""
    n_sfd = int((brim0 >= 0).sum())
    x_sfd = np.empty((n_sfd,) + x.shape[1:], dtype=x.dtype)
    Nd, T = brim0.shape
    for d in range(Nd):
        for t in range(T):
            v = brim0[d, t]
            if v >= 0:
                x_sfd[v] = x[t]
    return x_sfd


def build_brim1(ids: np.ndarray, local_experts: np.ndarray, row_tokens: np.ndarray) -> np.ndarray:
    """Algorithm 5 on one device.

    ``local_experts`` [n_loc] is the device's expert list L_loc (placement order);
    ``row_tokens`` [n_rows] is the ORI token of each received SFD row.  BRIM1[e, r]
    is a running counter taken expert by expert, row by row, over the (e, r) pairs
    whose row activates L_loc[e], and -1 elsewhere.  Returns int64 [n_loc, n_rows].
    """
    n_loc = len(local_experts)
    n_rows = len(row_tokens)
    chosen = [set(int(e) for e in ids[t]) for t in row_tokens]
    brim1 = np.empty((n_loc, n_rows), dtype=np.int64)
    ctr = 0
    for e in range(n_loc):
        for r in range(n_rows):
            if int(local_experts[e]) in chosen[r]:
                brim1[e, r] = ctr
                ctr += 1
            else:
                brim1[e, r] = -1
    return brim1


class Brims:
    """Every index structure of one layer call, built literally from Alg. 3 and 5."""

    def __init__(self, ids: np.ndarray, gates: np.ndarray, placement: np.ndarray):
        ids = np.asarray(ids)
        placement = np.asarray(placement)
        Nd, n_loc = placement.shape
        T, k = ids.shape
        e2v = np.empty(Nd * n_loc, dtype=np.int64)
        for d in range(Nd):
            for j in range(n_loc):
                e2v[placement[d, j]] = d
        act = np.zeros((T, Nd), dtype=bool)
        for t in range(T):
            for e in ids[t]:
                act[t, e2v[e]] = True
        self.placement = placement
        self.T, self.k, self.Nd, self.n_loc = T, k, Nd, n_loc
        self.brim0 = build_brim0(act)
        self.seg_off, self.row_tokens = segments(self.brim0)
        self.n_sfd = int(self.seg_off[-1])
        self.ct = act.sum(axis=1)
        self.brim1 = [build_brim1(ids, placement[d], self.row_tokens[d]) for d in range(Nd)]
        # global EPD layout implied by the per-device BRIM1 counters
        self.epd_base = np.zeros(Nd + 1, dtype=np.int64)
        for d in range(Nd):
            self.epd_base[d + 1] = self.epd_base[d] + int((self.brim1[d] >= 0).sum())
        n_epd = int(self.epd_base[-1])
        self.n_epd = n_epd
        self.epd_src = np.full(n_epd, -1, dtype=np.int64)    # SFD row feeding each EPD row
        self.epd_tok = np.full(n_epd, -1, dtype=np.int64)    # ORI token of each EPD row
        self.epd_exp = np.full(n_epd, -1, dtype=np.int64)    # expert of each EPD row
        self.epd_gate = np.zeros(n_epd, dtype=np.float64)
        self.exp_off = np.zeros(Nd * n_loc + 1, dtype=np.int64)  # per placement slot d*n_loc+j
        gate_of = {}
        for t in range(T):
            for j in range(k):
                gate_of[(t, int(ids[t, j]))] = gates[t, j]
        for d in range(Nd):
            b1 = self.brim1[d]
            for j in range(n_loc):
                e = int(placement[d, j])
                s = d * n_loc + j
                # rows of BRIM1 are numbered expert-major, so expert row j starts
                # after every entry of rows 0..j-1 (this holds for empty rows too)
                self.exp_off[s] = self.epd_base[d] + int((b1[:j] >= 0).sum())
                for r in range(b1.shape[1]):
                    v = b1[j, r]
                    if v >= 0:
                        g = self.epd_base[d] + v
                        t = int(self.row_tokens[d][r])
                        self.epd_src[g] = self.seg_off[d] + r
                        self.epd_tok[g] = t
                        self.epd_exp[g] = e
                        self.epd_gate[g] = gate_of[(t, e)]
        self.exp_off[-1] = n_epd

    def expert_to_vdev(self) -> np.ndarray:
        e2v = np.empty(self.Nd * self.n_loc, dtype=np.int64)
        for d in range(self.Nd):
            for j in range(self.n_loc):
                e2v[self.placement[d, j]] = d
        return e2v


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def occult_forward_staged(x: np.ndarray, ids: np.ndarray, gates: np.ndarray,
                          placement: np.ndarray, w1: np.ndarray, w2: np.ndarray,
                          brims: Brims = None):
    """The refactored pipeline of Algorithm 2, stage by stage, in fp64.

    dispatch (Alg. 4) -> all_to_all_0 (receive segment) -> scattering SMM with
    SwiGLU (Alg. 6) -> weight modulation (Alg. 7) -> merging SMM (Alg. 8, summing
    each SFD row's local experts) -> all_to_all_1 -> combine (Alg. 9, devices in
    order 0..Nd-1).  ``w1`` [Ne, 2I, d] (gate rows then up rows), ``w2`` [Ne, d, I].
    Returns ``y`` [T, d] and a dict of the intermediate tensors.
    """
    if brims is None:
        brims = Brims(ids, gates, placement)
    x = np.asarray(x, dtype=np.float64)
    w1 = np.asarray(w1, dtype=np.float64)
    w2 = np.asarray(w2, dtype=np.float64)
    I = w1.shape[1] // 2
    D = x.shape[1]
    x_sfd = dispatch(x, brims.brim0)
    h_epd = np.zeros((brims.n_epd, I), dtype=np.float64)
    y_epd = np.zeros((brims.n_epd, D), dtype=np.float64)
    y_sfd = np.zeros((brims.n_sfd, D), dtype=np.float64)
    for d in range(brims.Nd):
        lo, hi = brims.seg_off[d], brims.seg_off[d + 1]
        xs = x_sfd[lo:hi]                      # device d's received rows
        b1 = brims.brim1[d]
        base = brims.epd_base[d]
        for j in range(brims.n_loc):
            e = int(placement[d, j])
            rows = np.nonzero(b1[j] >= 0)[0]
            if rows.size == 0:
                continue
            a = xs[rows]
            g = a @ w1[e, :I].T
            u = a @ w1[e, I:].T
            dst = base + b1[j, rows]           # scatter to EPD rows
            h_epd[dst] = silu(g) * u
            # weight modulation with the token's gate for expert e
            h_epd[dst] *= brims.epd_gate[dst][:, None]
            y_epd[dst] = h_epd[dst] @ w2[e].T
        # merging: each SFD row sums its local experts' outputs (stage one)
        for j in range(brims.n_loc):
            rows = np.nonzero(b1[j] >= 0)[0]
            y_sfd[lo + rows] += y_epd[base + b1[j, rows]]
    # combine (stage two): sequential over devices
    y = np.zeros((brims.T, D), dtype=np.float64)
    for d in range(brims.Nd):
        for t in range(brims.T):
            v = brims.brim0[d, t]
            if v >= 0:
                y[t] += y_sfd[v]
    return y, {"x_sfd": x_sfd, "h_epd": h_epd, "y_epd": y_epd, "y_sfd": y_sfd}
