"""Sharded-source expert parallelism (oracle): every source device dispatches its
own tokens, and the first all-to-all is a real exchange of row blocks.

Test infrastructure: only the tests, the smoke check and the benchmark's CPU
baseline use this package; the CUDA library shares no code with it.

Occult paper, App. A.1-A.2: Algorithm 2 runs on every device of an
expert-parallel group; each device builds BRIM0 over its own N_ori tokens
(Algorithm 3) and dispatches them into its SFD tensor (Algorithm 4), whose
segment d goes to device d through all_to_all_single with the non-zero counts
of BRIM0 row d as split sizes (the text after Algorithm 4).  Here the T tokens
of one batch are split into n_src contiguous source shards [src_off[s],
src_off[s+1]) that stand for the source devices:

* send layout: shard s's SFD tensor follows shards 0..s-1; inside it, rows are
  device-major and in token order (Algorithm 3 over the shard's tokens);
* receive layout: device d receives the blocks of every source in source order,
  which for contiguous shards is exactly the single-source SFD layout (device-
  major over all T tokens in token order), so everything after the first
  exchange -- BRIM1, the expert GEMMs, stage one of the merge -- is unchanged;
* the second all-to-all returns device d's stage-one rows of source s to that
  source's send layout, and stage two sums a token's rows there.

Block (s, d) holds counts[s, d] rows: at send_off[s, d] in the send layout and
at recv_off[s, d] in the receive layout.
"""
from __future__ import annotations

from typing import Sequence

import numpy as np

from .brim import build_brim0


def shard_plan(act: np.ndarray, src_off: Sequence[int]):
    """``act`` [T, Nd] bool (token t uses device d), ``src_off`` [n_src + 1].

    Returns brim0_send int64 [Nd, T] (row of (d, t) in the send layout, -1 where
    inactive) and counts, send_off, recv_off, each int64 [n_src, Nd].
    """
    act = np.asarray(act, dtype=bool)
    T, Nd = act.shape
    src_off = [int(v) for v in src_off]
    n_src = len(src_off) - 1
    counts = np.zeros((n_src, Nd), dtype=np.int64)
    send_off = np.zeros((n_src, Nd), dtype=np.int64)
    recv_off = np.zeros((n_src, Nd), dtype=np.int64)
    brim0_send = np.full((Nd, T), -1, dtype=np.int64)
    base = 0
    for s in range(n_src):
        a, b = src_off[s], src_off[s + 1]
        local = build_brim0(act[a:b])           # Algorithm 3 on the shard's tokens
        brim0_send[:, a:b] = np.where(local >= 0, local + base, -1)
        counts[s] = act[a:b].sum(axis=0)
        send_off[s] = base + np.concatenate(([0], np.cumsum(counts[s])[:-1]))
        base += int(counts[s].sum())
    seg = np.concatenate(([0], np.cumsum(act.sum(axis=0))[:-1]))
    for s in range(n_src):
        recv_off[s] = seg + counts[:s].sum(axis=0)
    return brim0_send, counts, send_off, recv_off


def all_to_all(src: np.ndarray, counts: np.ndarray, send_off: np.ndarray,
               recv_off: np.ndarray, reverse: bool = False) -> np.ndarray:
    """The exchange as block copies: send -> receive layout, or back with ``reverse``."""
    out = np.zeros_like(src)
    n_src, Nd = counts.shape
    for s in range(n_src):
        for d in range(Nd):
            n = int(counts[s, d])
            a, b = (int(recv_off[s, d]), int(send_off[s, d])) if reverse else \
                   (int(send_off[s, d]), int(recv_off[s, d]))
            out[b:b + n] = src[a:a + n]
    return out
