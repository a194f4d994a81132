"""The Occult MoE layer forward, Algorithm 2 of the paper, as a sequence of C-ABI calls.

``OccultMoE`` owns the layer's weights, its expert placement and every buffer
of the pipeline, sized for the worst case so that no step waits on the host:

    route -> build BRIMs -> dispatch (ORI -> SFD, first all-to-all's send buffer)
    -> expert_up (SFD -> EPD, SwiGLU, modulation) -> [shared experts]
    -> expert_down_merge (the second linear layer; its rows added into the
       token rows with fp32 atomics, the paper's merging SMM)

or, with ``merge="ordered"`` (bit-reproducible), the down-projection writes the
fp32 EPD rows and ``combine`` sums them in a fixed order (EPD -> SFD -> ORI).

With ``src_off`` (contiguous source shards standing for the source devices of
App. A.1) the two all-to-alls are real exchanges of row blocks:

    route -> build BRIMs -> shard plan -> dispatch into the sources' send layout
    -> all_to_all (send -> receive) -> expert_up -> expert_down -> [shared]
    -> merge_sfd (stage one) -> all_to_all back (receive -> send)
    -> combine_sfd (stage two over each token's rows at its source)

PyTorch only allocates the buffers and provides the stream; all work runs in
the library's kernels.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import torch

from . import (MAX_SOURCES, OCCULT_BF16, OCCULT_F32, ROUTE_DEVICE_LIMITED, ROUTE_EXACT,
               ROUTE_SCORE_PRUNED, ROUTE_SIMILARITY_PRUNED, WS_BUILD_BRIM, WS_EXPERT_BWD,
               occult_all_to_all, occult_build_brim, occult_combine, occult_combine_sfd,
               occult_desc_t, occult_dispatch, occult_dispatch_epd, occult_expert_bwd,
               occult_expert_down,
               occult_expert_down_merge, occult_expert_bwd_merge,
               occult_expert_up, occult_gate_grad, occult_merge_sfd, occult_route,
               occult_route_similarity, occult_router_grad, occult_shard_plan,
               occult_shared_ffn, epd_copy_rows, workspace_size)


def desc_for(cfg, T: Optional[int] = None) -> occult_desc_t:
    """Descriptor from any object with the layer-config attribute names."""
    ds = occult_desc_t()
    ds.T = cfg.T if T is None else T
    ds.d = cfg.d
    ds.n_experts = cfg.n_experts
    ds.top_k = cfg.top_k
    ds.inter = cfg.inter
    ds.n_vdev = cfg.n_vdev
    ds.dtype = OCCULT_BF16 if cfg.dtype == "bf16" else OCCULT_F32
    ds.route_mode = {"exact": ROUTE_EXACT, "device_limited": ROUTE_DEVICE_LIMITED,
                     "score_pruned": ROUTE_SCORE_PRUNED,
                     "similarity_pruned": ROUTE_SIMILARITY_PRUNED}[cfg.route_mode]
    ds.limit_devices = cfg.limit_devices
    ds.renorm = int(bool(cfg.renorm))
    ds.n_shared = cfg.n_shared
    ds.shared_inter = cfg.shared_inter
    ds.shared_gate = int(bool(cfg.shared_gate))
    return ds


class OccultMoE:
    """One MoE layer resident on a CUDA device."""

    def __init__(self, desc: occult_desc_t, weights: Dict[str, torch.Tensor],
                 placement: torch.Tensor, device="cuda", materialize_sfd: bool = False,
                 train: bool = False, sim_table: Optional[torch.Tensor] = None,
                 src_off: Optional[Sequence[int]] = None, merge: Optional[str] = None):
        """``merge``: "atomic" (default; fp32 atomic adds into the token rows) or
        "ordered" (fixed order, bit-reproducible; the only one with a
        materialised SFD stage or source shards, and their default)."""
        self.desc = desc
        staged = materialize_sfd or src_off is not None
        if merge is None:
            merge = "ordered" if staged else "atomic"
        if merge not in ("atomic", "ordered") or (merge == "atomic" and staged):
            raise ValueError("merge must be 'ordered' or 'atomic'; the atomic merge has no "
                             "materialised SFD stage and no source shards")
        self.merge = merge
        if desc.route_mode == ROUTE_SIMILARITY_PRUNED and sim_table is None:
            raise ValueError("similarity-based pruning needs sim_table [Ne, Ne] (fp32)")
        dev = torch.device(device)
        dt = desc.torch_dtype
        self.device = dev
        self.w = {k: v.to(dev, dt).contiguous() for k, v in weights.items()}
        placement = torch.as_tensor(placement, dtype=torch.int32)
        # the kernels index by the placement without checking it (it lives in
        # device memory): it must hold every expert exactly once
        n_loc = desc.n_experts // max(1, desc.n_vdev)
        if (tuple(placement.shape) != (desc.n_vdev, n_loc)
                or sorted(placement.reshape(-1).tolist()) != list(range(desc.n_experts))):
            raise ValueError(f"placement must be [{desc.n_vdev}, {n_loc}] holding every one of "
                             f"the {desc.n_experts} experts exactly once")
        e2v = torch.empty(desc.n_experts, dtype=torch.int32)
        for d in range(placement.shape[0]):
            for e in placement[d].tolist():
                e2v[e] = d
        self.placement = placement.reshape(-1).to(dev).contiguous()
        self.expert_to_vdev = e2v.to(dev)
        T, d, Ne, k, Nd, I = desc.T, desc.d, desc.n_experts, desc.top_k, desc.n_vdev, desc.inter
        n_sfd_max = T * min(k, Nd)
        i32, f32 = torch.int32, torch.float32
        e = lambda *s, dtype=i32: torch.empty(*s, dtype=dtype, device=dev)  # noqa: E731
        self.ids, self.gates, self.vmask = e(T, k), e(T, k, dtype=f32), e(T)
        self.sim_table = (sim_table.to(dev, f32).contiguous() if sim_table is not None else None)
        # the experts whose probabilities the gates are (differs from ids only
        # under similarity-based pruning)
        self.routed = e(T, k) if desc.route_mode == ROUTE_SIMILARITY_PRUNED else self.ids
        self.logits = None
        self.brim0, self.seg_off, self.brim1 = e(Nd, T), e(Nd + 1), e(Ne, T)
        self.exp_off, self.epd_src, self.epd_gate = e(Ne + 1), e(T * k), e(T * k, dtype=f32)
        self.counts = e(4)
        self.brim_ws = e(max(1, workspace_size(desc, WS_BUILD_BRIM)), dtype=torch.uint8)
        self.x_sfd, self.sfd_tok = e(n_sfd_max, d, dtype=dt), e(n_sfd_max)
        # after the second linear layer everything is fp32
        self.h_epd = e(T * k, I, dtype=dt)
        self.y_epd = e(T * k, d, dtype=f32) if merge == "ordered" else None
        self.y = e(T, d, dtype=f32)
        self.y_sfd = e(n_sfd_max, d, dtype=f32) if materialize_sfd else None
        self.train = train
        if train:
            # forward saves G|U; backward buffers (weight gradients are fp32)
            self.gu_epd = e(T * k, 2 * I, dtype=dt)
            # the forward's gathered x rows and the backward's gathered dy rows in
            # padded EPD order, so that the weight gradients read them as tiles
            self.x_epd = e(epd_copy_rows(desc), d, dtype=dt)
            self.dy_epd = e(epd_copy_rows(desc), d, dtype=dt)
            # dy's SFD rows only with source shards (one source: dy goes straight
            # to dy_epd)
            self.dy_sfd = e(n_sfd_max, d, dtype=dt) if src_off is not None else None
            self.dgu_epd = e(T * k, 2 * I, dtype=dt)
            # fp32 EPD rows of dx only for the ordered merge
            self.dx_epd = e(T * k, d, dtype=f32) if merge == "ordered" else None
            self.dw1 = e(Ne, 2 * I, d, dtype=f32)
            self.dw2 = e(Ne, d, I, dtype=f32)
            self.dg_epd = e(T * k, dtype=f32)
            self.dgates = e(T, k, dtype=f32)
            self.dx = e(T, d, dtype=f32)
            self.dlogits = e(T, Ne, dtype=f32)
            self.bwd_ws = e(max(1, workspace_size(desc, WS_EXPERT_BWD)), dtype=torch.uint8)
        else:
            self.gu_epd = self.x_epd = None
        # sharded-source mode: the sources' send layout and the exchange plan
        self.src_off = None if src_off is None else [int(v) for v in src_off]
        if self.src_off is not None:
            n_src = len(self.src_off) - 1
            if not (1 <= n_src <= MAX_SOURCES) or self.src_off[0] != 0 or self.src_off[-1] != T:
                raise ValueError("src_off must run from 0 to T over 1..32 shards")
            self.n_src = n_src
            self.brim0_send = e(Nd, T)
            self.blk_counts, self.send_off, self.recv_off = e(n_src, Nd), e(n_src, Nd), e(n_src, Nd)
            self.x_send = e(n_sfd_max, d, dtype=dt)
            if self.y_sfd is None:
                self.y_sfd = e(n_sfd_max, d, dtype=f32)
            self.y_send = e(n_sfd_max, d, dtype=f32)
        if desc.n_shared:
            S = desc.n_shared * desc.shared_inter
            self.h_s, self.y_s = e(T, S, dtype=dt), e(T, d, dtype=f32)
            self.s_gate = e(T, dtype=f32)
        else:
            self.h_s = self.y_s = self.s_gate = None

    @property
    def launches_per_forward(self) -> int:
        """Kernels this object launches per forward call."""
        n = 8  # route, 3 BRIM kernels, dispatch, up, down, combine
        if self.merge == "atomic" and self.desc.n_shared:
            n -= 1  # the down-projection merges into the shared experts' output
        # (without shared experts the combine's place is taken by the zeroing of y)
        if self.src_off is not None:
            n += 4  # 2 plan kernels, 2 exchanges; combine runs as stage one + stage two
        if self.y_sfd is not None:
            n += 1
        if self.desc.n_shared:
            n += 2 + (1 if self.desc.shared_gate else 0)
        return n

    def route_and_index(self, logits: torch.Tensor, stream=None) -> None:
        ds = self.desc
        self.logits = logits
        if ds.route_mode == ROUTE_SIMILARITY_PRUNED:
            occult_route_similarity(ds, logits, self.expert_to_vdev, self.sim_table, self.ids,
                                    self.gates, self.vmask, self.routed, stream)
        else:
            occult_route(ds, logits, self.expert_to_vdev, self.ids, self.gates, self.vmask,
                         stream)
        occult_build_brim(ds, self.ids, self.gates, self.vmask, self.placement, self.brim0,
                          self.seg_off, self.brim1, self.exp_off, self.epd_src, self.epd_gate,
                          self.counts, self.brim_ws, stream)
        if self.src_off is not None:
            occult_shard_plan(ds, self.src_off, self.vmask, self.brim0, self.brim0_send,
                              self.blk_counts, self.send_off, self.recv_off, stream)

    def _scatter(self, src: torch.Tensor, out_sfd: torch.Tensor, sfd_tok, stream) -> None:
        """Stage one of scattering (Algorithm 4) and, sharded, the first all-to-all."""
        ds = self.desc
        if self.src_off is None:
            occult_dispatch(ds, src, self.brim0, self.vmask, out_sfd, sfd_tok, stream)
            return
        occult_dispatch(ds, src, self.brim0_send, self.vmask, self.x_send, None, stream)
        occult_all_to_all(ds, self.n_src, self.blk_counts, self.send_off, self.recv_off,
                          self.x_send, out_sfd, reverse=False, stream=stream)

    def _merge(self, y_epd: torch.Tensor, out: torch.Tensor, y_shared, stream) -> None:
        """The two-stage merge; sharded, the second all-to-all runs between the stages."""
        ds = self.desc
        if self.src_off is None:
            occult_combine(ds, y_epd, self.brim0, self.seg_off, self.brim1, self.exp_off, out,
                           y_shared=y_shared, y_sfd=self.y_sfd, stream=stream)
            return
        occult_merge_sfd(ds, y_epd, self.brim0, self.seg_off, self.brim1, self.exp_off,
                         self.y_sfd, stream)
        occult_all_to_all(ds, self.n_src, self.blk_counts, self.send_off, self.recv_off,
                          self.y_sfd, self.y_send, reverse=True, stream=stream)
        occult_combine_sfd(ds, self.y_send, self.brim0_send, out, y_shared=y_shared,
                           stream=stream)

    def forward(self, logits: torch.Tensor, x: torch.Tensor, stream=None,
                out: Optional[torch.Tensor] = None) -> torch.Tensor:
        """y = MoE(x) (fp32 [T, d]) for router logits ``logits`` [T, Ne] (fp32) and x [T, d].

        ``out``: an fp32 [T, d] CUDA tensor to write y into (default: the layer's own
        buffer), e.g. one of two alternating outputs whose device-to-host copy
        overlaps the next call."""
        ds = self.desc
        y = self.y if out is None else out
        if out is not None and (out.dtype != torch.float32 or out.numel() < ds.T * ds.d
                                or not out.is_contiguous()):
            raise ValueError("out must be a contiguous fp32 tensor of T * d elements")
        self.route_and_index(logits, stream)
        self._scatter(x, self.x_sfd, self.sfd_tok, stream)
        occult_expert_up(ds, self.x_sfd, self.epd_src, self.epd_gate, self.exp_off,
                         self.placement, self.w["w1"], self.h_epd, self.gu_epd, self.x_epd,
                         stream)
        if self.merge == "atomic":
            # the shared experts write y, the routed experts' rows are added to it
            if ds.n_shared:
                occult_shared_ffn(ds, x, self.w["ws1"], self.w["ws2"], self.w.get("w_sg"),
                                  self.h_s, self.s_gate, y, stream)
            occult_expert_down_merge(ds, self.h_epd, self.exp_off, self.placement, self.w["w2"],
                                     self.epd_src, self.sfd_tok, y,
                                     zero_y=not ds.n_shared, stream=stream)
            return y
        occult_expert_down(ds, self.h_epd, self.exp_off, self.placement, self.w["w2"],
                           self.y_epd, stream)
        if ds.n_shared:
            occult_shared_ffn(ds, x, self.w["ws1"], self.w["ws2"], self.w.get("w_sg"), self.h_s,
                              self.s_gate, self.y_s, stream)
        self._merge(self.y_epd, y, self.y_s, stream)
        return y

    @property
    def launches_per_backward(self) -> int:
        """Kernels one backward call launches."""
        # dispatch of dy (one source: to its padded EPD rows), 2 dgrad GEMMs, dg
        # reduce, 2 wgrad GEMMs, combine, gate grad,
        # router grad (+ 2 exchanges and the split merge when sharded)
        # (atomic merge: the dgrad through [W_g; W_u] merges dx, and the zeroing of
        # dx takes the combine's place)
        n = 9 + (1 if self.y_sfd is not None else 0)
        return n + (2 if self.src_off is not None else 0)

    def backward(self, dy: torch.Tensor, stream=None):
        """Gradients of sum(dy * y) after `forward` (train=True): (dx, dw1, dw2, dgates);
        the gradient of the router logits is left in ``self.dlogits`` [T, Ne].

        dy [T, d] in the layer dtype.  With one source the exchange is the
        identity, so dy goes in one pass to the padded EPD rows (BRIM0 -> BRIM1)
        that the backward GEMMs read as tiles; with source shards stage one sends
        it to the SFD rows and the first exchange moves them.  The expert backward
        runs on the EPD rows, and the two-stage merge brings dx back to the
        tokens; dgates return through BRIM0 -> BRIM1 as well, and on through the
        softmax of Eq. 2 to the logits the forward was given.
        """
        if not self.train:
            raise RuntimeError("OccultMoE was built without train=True")
        ds = self.desc
        if ds.n_shared:
            raise NotImplementedError("backward of shared experts is not provided")
        if self.src_off is None:
            occult_dispatch_epd(ds, dy, self.ids, self.placement, self.brim0, self.seg_off,
                                self.brim1, self.exp_off, self.dy_epd, stream)
        else:
            self._scatter(dy, self.dy_sfd, None, stream)
        if self.merge == "atomic":
            occult_expert_bwd_merge(ds, self.x_sfd, self.dy_sfd, self.epd_src, self.epd_gate,
                                    self.exp_off, self.placement, self.w["w1"], self.w["w2"],
                                    self.h_epd, self.gu_epd, self.dgu_epd, self.sfd_tok, self.dx,
                                    self.dw1, self.dw2, self.dg_epd, self.bwd_ws, self.x_epd,
                                    self.dy_epd, stream)
        else:
            self._expert_bwd_ordered(stream)
        occult_gate_grad(ds, self.ids, self.placement, self.brim0, self.seg_off, self.brim1,
                         self.exp_off, self.dg_epd, self.dgates, stream)
        occult_router_grad(ds, self.logits, self.routed, self.dgates, self.dlogits, stream)
        return self.dx, self.dw1, self.dw2, self.dgates

    def _expert_bwd_ordered(self, stream) -> None:
        ds = self.desc
        occult_expert_bwd(ds, self.x_sfd, self.dy_sfd, self.epd_src, self.epd_gate, self.exp_off,
                          self.placement, self.w["w1"], self.w["w2"], self.h_epd, self.gu_epd,
                          self.dgu_epd, self.dx_epd, self.dw1, self.dw2, self.dg_epd, self.bwd_ws,
                          self.x_epd, self.dy_epd, stream)
        self._merge(self.dx_epd, self.dx, None, stream)
