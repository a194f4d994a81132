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

    def oracle_route(self):
        cfg = self.cfg
        lg = self.logits.numpy()
        if cfg.route_mode == "device_limited":
            ids, gates, kept, margin = orouting.route_device_limited(
                lg, cfg.top_k, self.e2v, cfg.n_vdev, cfg.limit_devices)
            return ids, gates, margin
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


# Per-element error bounds of intermediates, derived from the arithmetic.  The
# 2e-2 * rms bar is the layer-output bar; the EPD intermediate h is heavy-tailed
# (a product silu(G) * U; max|h| reaches ~45 rms), so its bf16 rounding alone
# exceeds 2e-2 * rms(h) although every element is as exact as bf16 allows.
BF16_HALF_ULP = 2.0 ** -8     # |round_bf16(v) - v| <= 2^-8 |v|
F32_EPS = 2.0 ** -24


def h_bound(a: np.ndarray, wg: np.ndarray, wu: np.ndarray, gate: float, h_ref: np.ndarray,
            layer_dtype: str) -> np.ndarray:
    """Bound on |h_gpu - h_ref| for one EPD row.

    G = W_g a and U = W_u a accumulate K = len(a) products in fp32: their error is
    at most 2 K 2^-24 sum|w||a| (twice the textbook gamma_K, for any internal
    ordering of the tensor-core sum).  silu has slope <= 1.1, so the fp32 value of
    h = g silu(G) U is off by at most g (1.1 |U| dG + |silu G| dU + 1.1 dG dU) plus
    a few fp32 roundings; bf16 layers then round h once more (2^-8 relative).
    """
    a = a.astype(np.float64)
    K = a.size
    dG = 2 * K * F32_EPS * (np.abs(wg) @ np.abs(a))
    dU = 2 * K * F32_EPS * (np.abs(wu) @ np.abs(a))
    G = wg.astype(np.float64) @ a
    U_abs = np.abs(wu.astype(np.float64) @ a)
    s_abs = np.abs(G / (1.0 + np.exp(-G)))
    d32 = abs(gate) * (1.1 * U_abs * dG + s_abs * dU + 1.1 * dG * dU) + 8 * F32_EPS * np.abs(h_ref)
    if layer_dtype == "f32":
        return d32
    return BF16_HALF_ULP * (np.abs(h_ref) + d32) + d32


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
