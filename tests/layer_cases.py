"""Seeded layer cases shared by the GPU parity tests, the smoke check and the
benchmark: inputs from ``synth``, placement and expected values from ``oracle``.

Nothing here calls the CUDA path; tensors destined for the GPU are produced on
the host (or drawn on the device by the seeded generator and copied back) and
the oracle always sees the same values.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np
import torch

import synth
from oracle import brim as obrim
from oracle import coact as ocoact
from oracle import expert as oexpert
from oracle import placement as oplace
from oracle import routing as orouting


@dataclasses.dataclass
class Case:
    cfg: synth.LayerConfig
    logits: torch.Tensor            # fp32 [T, Ne], CPU
    x: torch.Tensor                 # [T, d] layer dtype, on `device`
    weights: Dict[str, torch.Tensor]  # layer dtype, on `device`
    placement: np.ndarray           # int32 [Nd, n_loc]

    @property
    def e2v(self) -> np.ndarray:
        return oplace.expert_to_vdev(self.placement)

    def host(self, name: str) -> np.ndarray:
        """A tensor as fp32 numpy (exact for bf16 values)."""
        t = self.x if name == "x" else self.weights[name]
        return t.detach().float().cpu().numpy()

    def oracle_route(self, table: Optional[np.ndarray] = None):
        """Oracle routing: ids, gates and the relative margin of a float decision
        (inf where none is taken); ``table`` for similarity-based pruning."""
        cfg = self.cfg
        lg = self.logits.numpy()
        if cfg.route_mode == "device_limited":
            ids, gates, kept, margin = orouting.route_device_limited(
                lg, cfg.top_k, self.e2v, cfg.n_vdev, cfg.limit_devices)
            return ids, gates, margin
        if cfg.route_mode == "score_pruned":
            ids, gates, _ = orouting.route_score_pruned(lg, cfg.top_k, self.e2v,
                                                        cfg.limit_devices, renorm=cfg.renorm)
            return ids, gates, np.full(lg.shape[0], np.inf)
        if cfg.route_mode == "similarity_pruned":
            ids, gates, _, _ = orouting.route_similarity_pruned(
                lg, cfg.top_k, self.e2v, cfg.limit_devices, table, renorm=cfg.renorm)
            return ids, gates, np.full(lg.shape[0], np.inf)
        ids, gates = orouting.route_topk(lg, cfg.top_k, renorm=cfg.renorm)
        return ids, gates, np.full(lg.shape[0], np.inf)


_placements: Dict[tuple, np.ndarray] = {}


def alg1_placement(cfg: synth.LayerConfig) -> np.ndarray:
    """Algorithm 1 on the profiling batch of the config (oracle, cached)."""
    key = (cfg.n_experts, cfg.top_k, cfg.n_vdev, cfg.n_clusters, cfg.experts_per_cluster,
           cfg.prof_tokens)
    if key not in _placements:
        ids, _ = orouting.route_topk(synth.profiling_logits(cfg).numpy(), cfg.top_k)
        _placements[key] = oplace.place(ocoact.coactivation(ids, cfg.n_experts), cfg.n_vdev)
    return _placements[key]


def make_case(cfg: synth.LayerConfig, T: Optional[int] = None, placement: str = "alg1",
              device="cuda", logits: Optional[torch.Tensor] = None, tensors: bool = True) -> Case:
    """A seeded case; ``tensors=False`` skips drawing x and the weights."""
    if T is not None:
        cfg = cfg.with_(T=T)
    if logits is None:
        logits = synth.measured_logits(cfg)
    gen_dev = device if torch.cuda.is_available() and str(device).startswith("cuda") else "cpu"
    x = synth.hidden_states(cfg, device=gen_dev) if tensors else None
    w = synth.expert_weights(cfg, device=gen_dev) if tensors else {}
    if placement == "alg1":
        L = alg1_placement(cfg)
    elif placement == "trivial":
        L = oplace.trivial(cfg.n_experts, cfg.n_vdev)
    else:
        rng = np.random.default_rng(7)
        L = rng.permutation(cfg.n_experts).reshape(cfg.n_vdev, -1).astype(np.int32)
    return Case(cfg, logits, x, w, np.asarray(L, dtype=np.int32))


def reference_output(case: Case, tokens, ids=None, gates=None) -> np.ndarray:
    """Oracle Eq. 1 layer output (plus shared experts) for a subset of tokens, fp64."""
    if ids is None:
        ids, gates, _ = case.oracle_route()
    x = case.host("x")
    w = {"w1": case.host("w1"), "w2": case.host("w2")}
    if "ws1" in case.weights:
        w["ws1"] = case.host("ws1")
        w["ws2"] = case.host("ws2")
        if "w_sg" in case.weights:
            w["w_sg"] = case.host("w_sg")
    return oexpert.layer_output(x, ids, gates, w, tokens)


def bf16_bar(ref: np.ndarray) -> float:
    """Layer-output tolerance for bf16 layers: max|diff| <= 2e-2 * rms(ref)."""
    return 2e-2 * float(np.sqrt(np.mean(np.square(ref))))


def assert_close_layer(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = "y") -> None:
    err = float(np.max(np.abs(got.astype(np.float64) - ref))) if ref.size else 0.0
    if dtype == "f32":
        # fp32 layers: max|diff| / max|ref| <= 1e-5
        scale = float(np.max(np.abs(ref))) if ref.size else 1.0
        assert err <= 1e-5 * scale, f"{what}: max|diff| {err:.3e} > 1e-5 * {scale:.3e}"
    else:
        bar = bf16_bar(ref)
        assert err <= bar, f"{what}: max|diff| {err:.3e} > 2e-2 * rms = {bar:.3e}"


def oracle_brims(case: Case, ids, gates) -> obrim.Brims:
    return obrim.Brims(ids, gates, case.placement)


def scatter_add_rows(dst: np.ndarray, idx: np.ndarray, rows: np.ndarray) -> None:
    """dst[idx[i]] += rows[i] for every i, repeated indices summed (rows sharing an
    index are added together first, in order, then once into dst)."""
    idx = np.asarray(idx, dtype=np.int64)
    if idx.size == 0:
        return
    order = np.argsort(idx, kind="stable")
    s_idx = idx[order]
    starts = np.concatenate([[0], np.nonzero(np.diff(s_idx))[0] + 1])
    dst[s_idx[starts]] += np.add.reduceat(rows[order], starts, axis=0)


# Per-element error bounds of intermediates, derived from the arithmetic.  The
# 2e-2 * rms bar is the layer-output bar; the EPD intermediate h is heavy-tailed
# (a product silu(G) * U; max|h| reaches ~45 rms), so its bf16 rounding alone
# exceeds 2e-2 * rms(h) although every element is as exact as bf16 allows.
BF16_HALF_ULP = 2.0 ** -8     # |round_bf16(v) - v| <= 2^-8 |v|
F32_EPS = 2.0 ** -24


def abs_contract(a_abs: np.ndarray, b_abs: np.ndarray) -> np.ndarray:
    """a_abs @ b_abs for non-negative matrices, as an upper bound: the product is
    taken in fp32 (fast) and raised by 1 %, which covers its own rounding (a sum
    of K non-negative fp32 terms, each rounded on the way in, is within
    (K + 2) 2^-24 of the exact value: under 1 % for K < 160000)."""
    r = np.asarray(a_abs, dtype=np.float32) @ np.asarray(b_abs, dtype=np.float32)
    return r.astype(np.float64) * 1.01


def h_bound(a: np.ndarray, wg: np.ndarray, wu: np.ndarray, gate, h_ref: np.ndarray,
            layer_dtype: str) -> np.ndarray:
    """Bound on |h_gpu - h_ref| for one EPD row (a [d], gate a scalar, h_ref [I]) or
    for several rows of one expert at once (a [n, d], gate [n], h_ref [n, I]).

    G = W_g a and U = W_u a accumulate K = d products in fp32: their error is at
    most 2 K 2^-24 sum|w||a| (twice the textbook gamma_K, for any internal
    ordering of the tensor-core sum).  silu has slope <= 1.1, so the fp32 value of
    h = g silu(G) U is off by at most g (1.1 |U| dG + |silu G| dU + 1.1 dG dU) plus
    a few fp32 roundings; bf16 layers then round h once more (2^-8 relative).
    """
    single = np.ndim(a) == 1
    a = np.atleast_2d(np.asarray(a, dtype=np.float64))
    wg = np.asarray(wg, dtype=np.float64)
    wu = np.asarray(wu, dtype=np.float64)
    g = np.abs(np.atleast_1d(np.asarray(gate, dtype=np.float64)))[:, None]
    h_ref = np.atleast_2d(h_ref)
    K = a.shape[1]
    aa = np.abs(a)
    dG = 2 * K * F32_EPS * abs_contract(aa, np.abs(wg).T)
    dU = 2 * K * F32_EPS * abs_contract(aa, np.abs(wu).T)
    G = a @ wg.T
    U_abs = np.abs(a @ wu.T)
    s_abs = np.abs(G / (1.0 + np.exp(-G)))
    d32 = g * (1.1 * U_abs * dG + s_abs * dU + 1.1 * dG * dU) + 8 * F32_EPS * np.abs(h_ref)
    out = d32 if layer_dtype == "f32" else BF16_HALF_ULP * (np.abs(h_ref) + d32) + d32
    return out[0] if single else out


def sfd_bound(w2: np.ndarray, h_abs_rows, layer_dtype: str) -> np.ndarray:
    """Bound on |y_sfd_gpu - y_sfd_ref| for one SFD row summing the given EPD rows.

    Each EPD row y = W_d h' reads h' rounded to the layer dtype (2^-8 relative for
    bf16, with the small fp32 error of h' folded in as 1 %), accumulates I products
    in fp32 (2 I 2^-24 sum|W||h'|), and the row sum adds one fp32 rounding per row.
    """
    B = 0.0
    for e, h_abs in h_abs_rows:
        B = B + np.abs(w2[e]).astype(np.float64) @ h_abs
    I = w2.shape[-1]
    rel = (1.01 * BF16_HALF_ULP if layer_dtype == "bf16" else 8 * F32_EPS)
    rel += (2 * I + 2 * len(h_abs_rows) + 4) * F32_EPS
    return rel * B


# Random-walk bounds.  The worst-case error of a sum of K terms, each carrying an
# independent rounding error e_i with |e_i| <= b_i, is sum b_i; the errors of
# round-to-nearest of distinct values behave as independent and zero-mean, and
# for such errors Hoeffding's inequality gives |sum e_i| <= LAMBDA sqrt(sum b_i^2)
# except with probability 2 exp(-LAMBDA^2 / 2) (4e-22 per element at 10).  The
# long reductions of dgates (over I) and dx (over 2I) use this form: their
# worst-case bounds are sqrt(K) times looser than the errors the arithmetic
# makes and would let a dropped EPD row pass.
LAMBDA = 10.0


def expert_backward_bounds(x, dy, w1e, w2e, gate, layer_dtype="bf16"):
    """Oracle-side intermediates and per-element error bounds of one expert's rows.

    x, dy [n, d] are the rows' token inputs and upstream gradients (exact bf16
    values), gate [n] their routing weights, w1e [2I, d], w2e [d, I].  The GPU
    saves G and U in bf16 in the forward, reads h' = g silu(G) U in bf16, rounds
    dG and dU to bf16 and accumulates every contraction in fp32.  Returns a dict
    with fp64 references and bounds:
      dG, dU, dG_b, dU_b [n, I]; dx_rows, dx_rows_b [n, d] (each row's W1^T dGU);
      dg, dg_b [n]; h1 (= h'), h1_b [n, I]; dW1_b [2I, d]; dW2_b [d, I].
    """
    f64 = np.float64
    x = np.asarray(x, f64)
    dy = np.asarray(dy, f64)
    wg = np.asarray(w1e, f64)[: w1e.shape[0] // 2]
    wu = np.asarray(w1e, f64)[w1e.shape[0] // 2:]
    wd = np.asarray(w2e, f64)
    g = np.asarray(gate, f64)[:, None]
    n, d = x.shape
    I = wg.shape[0]
    u = BF16_HALF_ULP
    acc = lambda K, m: 2 * K * F32_EPS * m  # noqa: E731  fp32 accumulation of K terms
    G = x @ wg.T
    U = x @ wu.T
    # fp32 accumulation of G and U over d terms, as a random walk (see dh' below)
    acc_rw = lambda K, m: LAMBDA * np.sqrt(K) * F32_EPS * m  # noqa: E731
    aG = acc_rw(d, abs_contract(np.abs(x), np.abs(wg).T))
    aU = acc_rw(d, abs_contract(np.abs(x), np.abs(wu).T))
    dG_st = aG * (1 + u) + u * np.abs(G)      # |stored bf16 G - G|
    dU_st = aU * (1 + u) + u * np.abs(U)
    sig = 1.0 / (1.0 + np.exp(-G))
    s = G * sig
    h1 = g * s * U
    h1_32 = np.abs(g) * (1.1 * np.abs(U) * aG + np.abs(s) * aU + 1.1 * aG * aU) + 8 * F32_EPS * np.abs(h1)
    h1_b = h1_32 * (1 + u) + u * np.abs(h1)
    dhp = dy @ wd
    # dh' = dy W_d: its fp32 accumulation error over d terms as a random walk
    # (Higham and Mary's probabilistic bound, LAMBDA sqrt(d) 2^-24 sum|terms|):
    # its worst case, 2 d 2^-24 sum|terms|, would dominate every bound below it
    ddhp = acc_rw(d, abs_contract(np.abs(dy), np.abs(wd)))
    ds = 1.1 * dG_st
    sU = s * U
    dg = np.sum(dhp * sU, axis=1)
    # dg sums I products whose errors come from independent roundings (fp32 sums
    # of other output columns, bf16 G and U of other units): a random-walk bound
    # on them (Hoeffding, LAMBDA), the fp32 sum of the products worst case
    dg_terms = ddhp * np.abs(sU) + np.abs(dhp) * (ds * np.abs(U) + np.abs(s) * dU_st + ds * dU_st)
    dg_b = (LAMBDA * np.sqrt(np.sum(dg_terms ** 2, axis=1))
            + acc(I, np.sum(np.abs(dhp * sU), axis=1)) + 1e-30)
    silu1 = sig * (1.0 + G * (1.0 - sig))
    dG = g * dhp * U * silu1
    dU = g * dhp * s
    dG_pre = np.abs(g) * (ddhp * np.abs(U * silu1) +
                          np.abs(dhp) * (1.1 * dU_st + 0.5 * np.abs(U) * dG_st + 0.5 * dG_st * dU_st))
    dG_pre += 8 * F32_EPS * np.abs(dG)
    dU_pre = np.abs(g) * (ddhp * np.abs(s) + np.abs(dhp) * ds) + 8 * F32_EPS * np.abs(dU)
    dG_b = dG_pre * (1 + u) + u * np.abs(dG)
    dU_b = dU_pre * (1 + u) + u * np.abs(dU)
    dx_rows = dG @ wg + dU @ wu
    dGa, dUa = np.abs(dG) + dG_b, np.abs(dU) + dU_b
    # each bound below is (rounding of the operands) + (fp32 accumulation of K
    # terms); both are contractions with the same absolute operand, so they are
    # summed before the one matrix product
    # a dx row contracts 2I values of dG | dU with independent rounding errors
    # (random-walk bound, LAMBDA) plus the worst-case fp32 accumulation
    dx_rows_b = (LAMBDA * np.sqrt(abs_contract(dG_b ** 2, wg ** 2) + abs_contract(dU_b ** 2, wu ** 2))
                 + abs_contract(acc(2 * I, dGa), np.abs(wg)) + abs_contract(acc(2 * I, dUa), np.abs(wu)))
    ax = np.abs(x)
    dW1_b = np.concatenate([abs_contract((dG_b + acc(n, dGa)).T, ax),
                            abs_contract((dU_b + acc(n, dUa)).T, ax)])
    dW2_b = abs_contract(np.abs(dy).T, h1_b + acc(n, np.abs(h1) + h1_b))
    return dict(dG=dG, dU=dU, dG_b=dG_b, dU_b=dU_b, dx_rows=dx_rows, dx_rows_b=dx_rows_b,
                dg=dg, dg_b=dg_b, h1=h1, h1_b=h1_b, dW1_b=dW1_b, dW2_b=dW2_b)
