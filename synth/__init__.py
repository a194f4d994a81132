"""Seeded synthetic inputs for the Occult MoE layer.

This module only draws random tensors; it holds none of the layer's arithmetic.
It is the one piece of code shared by the CPU oracle's callers (tests, the
benchmark's CPU baseline) and the CUDA path's callers: both sides are handed
the very same tensors.

Workload recipe (the pages measure real OLMoE / Qwen1.5-MoE / DeepSeek-MoE
checkpoints on real data; these seeded stand-ins keep their shapes, k and Ne):

* hidden states ``x ~ N(0, 1)``;
* every expert weight ``~ N(0, 0.02^2)`` (standard deviation 0.02);
* router logits ``= N(0, 1) + 3 * A[c_t, e]`` where each token draws a latent
  cluster ``c_t ~ Uniform{0..C-1}`` and ``A`` is a 0/1 cluster-to-expert mask
  with ``m`` distinct experts per cluster, drawn without replacement.  The same
  ``A`` (seed 1000) serves the profiling batch (seed 1003) and the measured
  batch (seed 1002), so a placement profiled on one transfers to the other;
* upstream gradient ``dy ~ N(0, 1)`` (seed 1004); weights use seed 1001.

Values are drawn in fp32 and rounded to nearest-even bf16 for bf16 layers.
Small tensors (logits, masks) are always drawn on the CPU, so routing is the
same on every machine.  Large tensors may be drawn on a CUDA device with a
seeded CUDA generator (a CPU draw of ~10^9 normals takes minutes); callers copy
them to the host for the oracle, so both sides still see identical values.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import torch

SEED_CLUSTERS = 1000
SEED_WEIGHTS = 1001
SEED_BATCH = 1002
SEED_PROFILE = 1003
SEED_DY = 1004
SEED_TABLE = 1005


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    """Shape and routing options of one MoE layer workload."""

    name: str
    T: int                     # tokens in the measured batch (N_ori)
    d: int                     # hidden size
    n_experts: int             # Ne
    top_k: int                 # k
    inter: int                 # SwiGLU intermediate size of a routed expert
    n_vdev: int                # Nd virtual expert-parallel devices
    dtype: str                 # "f32" or "bf16"
    n_clusters: int            # latent token clusters C
    experts_per_cluster: int   # m experts boosted per cluster
    prof_tokens: int           # tokens in the profiling batch
    renorm: bool = False       # renormalise the k gates to sum to one
    # "exact", "device_limited" (gate mass), or the pages' own rules
    # "score_pruned" and "similarity_pruned"
    route_mode: str = "exact"
    limit_devices: int = 2     # devices kept in device-limited mode
    n_shared: int = 0          # always-on shared experts
    shared_inter: int = 0      # intermediate size of each shared expert
    shared_gate: bool = False  # sigmoid(w_sg . x) gate on the shared output
    backward: bool = False     # the workload includes the backward pass
    n_src: int = 1             # source shards (1: the whole batch is one source)

    @property
    def n_loc(self) -> int:
        return self.n_experts // self.n_vdev

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_(self, **kw) -> "LayerConfig":
        return dataclasses.replace(self, **kw)


CONFIGS: Dict[str, LayerConfig] = {
    # tiny fp32 layer
    "tiny_f32": LayerConfig("tiny_f32", T=256, d=64, n_experts=8, top_k=2, inter=128,
                            n_vdev=4, dtype="f32", n_clusters=4, experts_per_cluster=3,
                            prof_tokens=1024, renorm=True),
    # OLMoE-shaped forward layer
    "olmoe_fwd": LayerConfig("olmoe_fwd", T=4096, d=2048, n_experts=64, top_k=8, inter=1024,
                             n_vdev=8, dtype="bf16", n_clusters=16, experts_per_cluster=10,
                             prof_tokens=16384),
    # Qwen1.5-MoE-A2.7B-shaped prefill layer with one sigmoid-gated shared expert
    "qwen_prefill": LayerConfig("qwen_prefill", T=16384, d=2048, n_experts=60, top_k=4,
                                inter=1408, n_vdev=4, dtype="bf16", n_clusters=12,
                                experts_per_cluster=8, prof_tokens=16384, n_shared=1,
                                shared_inter=5632, shared_gate=True),
    # DeepSeek-MoE-16B-shaped decode layer with two ungated shared experts
    "deepseek_decode": LayerConfig("deepseek_decode", T=512, d=2048, n_experts=64, top_k=6,
                                   inter=1408, n_vdev=8, dtype="bf16", n_clusters=16,
                                   experts_per_cluster=10, prof_tokens=16384, n_shared=2,
                                   shared_inter=1408),
    # the same decode layer with device-limited routing: the 2 virtual devices of
    # largest gate mass, renormalised top-k among their experts
    "deepseek_decode_limited": LayerConfig("deepseek_decode_limited", T=512, d=2048,
                                           n_experts=64, top_k=6, inter=1408, n_vdev=8,
                                           dtype="bf16", n_clusters=16, experts_per_cluster=10,
                                           prof_tokens=16384, n_shared=2, shared_inter=1408,
                                           route_mode="device_limited", renorm=True),
    # the OLMoE-shaped forward under the pages' collaboration pruning to 2 devices
    "olmoe_fwd_score_pruned": LayerConfig("olmoe_fwd_score_pruned", T=4096, d=2048,
                                          n_experts=64, top_k=8, inter=1024, n_vdev=8,
                                          dtype="bf16", n_clusters=16, experts_per_cluster=10,
                                          prof_tokens=16384, route_mode="score_pruned"),
    "olmoe_fwd_similarity_pruned": LayerConfig("olmoe_fwd_similarity_pruned", T=4096, d=2048,
                                               n_experts=64, top_k=8, inter=1024, n_vdev=8,
                                               dtype="bf16", n_clusters=16,
                                               experts_per_cluster=10, prof_tokens=16384,
                                               route_mode="similarity_pruned"),
    # the OLMoE-shaped forward with the batch split over 8 source devices: the
    # first all-to-all is a real exchange of row blocks (and the second its reverse)
    "olmoe_fwd_sharded": LayerConfig("olmoe_fwd_sharded", T=4096, d=2048, n_experts=64,
                                     top_k=8, inter=1024, n_vdev=8, dtype="bf16",
                                     n_clusters=16, experts_per_cluster=10, prof_tokens=16384,
                                     n_src=8),
    # OLMoE-shaped training step (forward + backward)
    "olmoe_train": LayerConfig("olmoe_train", T=32768, d=2048, n_experts=64, top_k=8,
                               inter=1024, n_vdev=16, dtype="bf16", n_clusters=16,
                               experts_per_cluster=10, prof_tokens=16384, backward=True),
}


def source_offsets(cfg: LayerConfig, n_tokens: Optional[int] = None):
    """Token offsets [n_src + 1] of ``cfg.n_src`` contiguous, near-equal source shards."""
    T = cfg.T if n_tokens is None else n_tokens
    return [s * T // cfg.n_src for s in range(cfg.n_src + 1)]


def cluster_mask(cfg: LayerConfig, seed: int = SEED_CLUSTERS) -> torch.Tensor:
    """0/1 mask A [C, Ne]: row c marks ``experts_per_cluster`` distinct experts."""
    g = torch.Generator().manual_seed(seed)
    A = torch.zeros(cfg.n_clusters, cfg.n_experts, dtype=torch.float32)
    for c in range(cfg.n_clusters):
        pick = torch.randperm(cfg.n_experts, generator=g)[: cfg.experts_per_cluster]
        A[c, pick] = 1.0
    return A


def router_logits(cfg: LayerConfig, n_tokens: int, seed: int,
                  A: Optional[torch.Tensor] = None) -> torch.Tensor:
    """fp32 logits [n_tokens, Ne] = N(0,1) + 3 * A[c_t]; always drawn on the CPU."""
    if A is None:
        A = cluster_mask(cfg)
    g = torch.Generator().manual_seed(seed)
    c = torch.randint(0, cfg.n_clusters, (n_tokens,), generator=g)
    noise = torch.randn(n_tokens, cfg.n_experts, generator=g, dtype=torch.float32)
    return (noise + 3.0 * A[c]).contiguous()


def _normal(shape, std: float, seed: int, dtype: torch.dtype, device) -> torch.Tensor:
    device = torch.device(device)
    g = torch.Generator(device=device).manual_seed(seed)
    out = torch.empty(shape, dtype=dtype, device=device)
    # draw in fp32 slabs to bound the temporary, then round to the target type
    flat = out.view(-1)
    slab = 1 << 26
    for i in range(0, flat.numel(), slab):
        n = min(slab, flat.numel() - i)
        v = torch.randn(n, generator=g, dtype=torch.float32, device=device)
        if std != 1.0:
            v.mul_(std)
        flat[i:i + n].copy_(v)
    return out


def hidden_states(cfg: LayerConfig, n_tokens: Optional[int] = None, seed: int = SEED_BATCH,
                  device="cpu") -> torch.Tensor:
    """x [T, d] ~ N(0, 1) in the layer dtype."""
    T = cfg.T if n_tokens is None else n_tokens
    return _normal((T, cfg.d), 1.0, seed * 7 + 1, cfg.torch_dtype, device)


def expert_weights(cfg: LayerConfig, seed: int = SEED_WEIGHTS, device="cpu") -> Dict[str, torch.Tensor]:
    """Routed and shared expert weights, all ~N(0, 0.02^2).

    * ``w1`` [Ne, 2*I, d]: rows [0, I) are the SwiGLU gate projection W_g, rows
      [I, 2I) the up projection W_u (each row is one output unit, K = d contiguous).
    * ``w2`` [Ne, d, I]: the down projection W_d (row = output unit, K = I contiguous).
    * shared experts (if any) are stacked along the intermediate axis:
      ``ws1`` [2*S, d] with S = n_shared * shared_inter (gate rows then up rows),
      ``ws2`` [d, S]; ``w_sg`` [d] is the sigmoid gate vector when enabled.
    """
    dt = cfg.torch_dtype
    out = {
        "w1": _normal((cfg.n_experts, 2 * cfg.inter, cfg.d), 0.02, seed * 7 + 2, dt, device),
        "w2": _normal((cfg.n_experts, cfg.d, cfg.inter), 0.02, seed * 7 + 3, dt, device),
    }
    if cfg.n_shared:
        S = cfg.n_shared * cfg.shared_inter
        out["ws1"] = _normal((2 * S, cfg.d), 0.02, seed * 7 + 4, dt, device)
        out["ws2"] = _normal((cfg.d, S), 0.02, seed * 7 + 5, dt, device)
        if cfg.shared_gate:
            out["w_sg"] = _normal((cfg.d,), 0.02, seed * 7 + 6, dt, device)
    return out


def upstream_grad(cfg: LayerConfig, n_tokens: Optional[int] = None, seed: int = SEED_DY,
                  device="cpu") -> torch.Tensor:
    """dy [T, d] ~ N(0, 1) in the layer dtype."""
    T = cfg.T if n_tokens is None else n_tokens
    return _normal((T, cfg.d), 1.0, seed * 7 + 5, cfg.torch_dtype, device)


def measured_logits(cfg: LayerConfig, n_tokens: Optional[int] = None) -> torch.Tensor:
    return router_logits(cfg, cfg.T if n_tokens is None else n_tokens, SEED_BATCH)


def profiling_logits(cfg: LayerConfig) -> torch.Tensor:
    return router_logits(cfg, cfg.prof_tokens, SEED_PROFILE)


def random_similarity_table(cfg: LayerConfig, seed: int = SEED_TABLE) -> torch.Tensor:
    """A seeded symmetric fp32 [Ne, Ne] table of values in [-1, 1] (diagonal 1), the
    shape of a similarity table, for checking pruning by similarity apart from how
    a table is built."""
    g = torch.Generator().manual_seed(seed)
    a = torch.rand(cfg.n_experts, cfg.n_experts, generator=g, dtype=torch.float32) * 2 - 1
    a = torch.triu(a, diagonal=1)
    return a + a.T + torch.eye(cfg.n_experts)
