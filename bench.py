"""Throughput of the Occult MoE layer (tokens/s) on GB300, with roofline and CPU baseline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config NAME]
                    [--merge atomic|ordered] [--tokens T]

One step = one training step of the layer (the default workload, ``olmoe_train``):
the forward path (route -> BRIM build -> dispatch -> grouped SwiGLU expert GEMMs
-> merge of the expert outputs) and its backward (dispatch of dy to its padded
EPD rows -> the four backward GEMMs -> gate and router-logit gradients) over one
batch of the OLMoE-shaped bf16 training workload (T=32768, d=2048, Ne=64, k=8,
I=1024, Nd=16 virtual devices), with the Algorithm 1 placement from a 16384-token
profiling batch computed through the library (the batch routed and its
co-activation counted on the GPU, Algorithm 1 on the host; reported under
"offline", not timed).  ``--config olmoe_fwd`` and the others time the forward
of the other workloads.  Inputs are resident in HBM when the timed region starts;
they are larger than L2 (the expert weights alone are 805 MB), so no L2 flush is
needed between steps.  The end-to-end figure runs the same steps through
OccultMoE.forward / backward with the inputs copied from pinned host memory and
the output read back every step.

Under torchrun (N > 1) every rank runs its own replica of the layer on its own
batch (the layer's batches are independent problems; no data-path collective),
so the scaling is weak.  Prints ONE JSON line on rank 0.

``--impl reference`` times the plain CPU oracle (the only reference of this
method) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "Occult MoE-layer tokens/s on 1 GB300"
UNIT = "tokens/s"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default="olmoe_train")
    p.add_argument("--merge", choices=["atomic", "ordered"], default=None,
                   help="merge of the expert outputs (default: atomic; ordered with source "
                        "shards)")
    p.add_argument("--tokens", type=int, default=None,
                   help="override the workload's token count (smaller profiling cases)")
    p.add_argument("--cpu-seconds", type=float, default=15.0,
                   help="CPU time of the oracle sample in the baseline leg")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_desc(cfg) -> str:
    s = (f"{cfg.name}: T={cfg.T} d={cfg.d} Ne={cfg.n_experts} k={cfg.top_k} I={cfg.inter} "
         f"Nd={cfg.n_vdev} {cfg.dtype} {cfg.route_mode}")
    if cfg.n_src > 1:
        s += f" n_src={cfg.n_src}"
    if cfg.n_shared:
        s += f" shared={cfg.n_shared}x{cfg.shared_inter}"
    return s + ", Algorithm 1 placement"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        else:
            self.lines = []

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], None, set()
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def peaks():
    """HBM GB/s, bf16 TFLOP/s burst and sustained, and where they come from."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return (j.get("hbm_gbs", 6800.0), j.get("bf16_tflops", 1900.0),
                j.get("bf16_tflops_sustained", 1700.0), "measured")
    return 6800.0, 1900.0, 1700.0, "fallback"


# A timed region this long keeps the GPU at its power limit like the sustained
# GEMM loop of the peak measurement (seconds back to back): its tensor kernels
# are graded against the sustained bf16 figure, shorter ones against the burst.
SUSTAINED_MS = 1000.0


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        j = json.load(f)
    e = j.get(workload, {}).get(kernel)
    if not e:
        return None
    src = os.path.join(ROOT, "combine_top_route_gb300", "csrc", e["source"])
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()[:16]
    return e["bytes_per_launch"] if h == e["source_sha256_16"] else None


class OracleSample:
    """The oracle as it stands, timed on the host cores on the first tokens of the batch."""

    def __init__(self, cfg):
        from layer_cases import alg1_placement
        self.cfg = cfg
        self.L = alg1_placement(cfg)
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        self.logits = synth.measured_logits(cfg).numpy()
        self.x = synth.hidden_states(cfg, device=dev).float().cpu().numpy()
        self.w = {k: v.float().cpu().numpy()
                  for k, v in synth.expert_weights(cfg, device=dev).items()}
        # a training workload's step is forward + backward on both sides
        self.dy = (synth.upstream_grad(cfg, device=dev).float().cpu().numpy()
                   if cfg.backward else None)
        capped = [int(os.environ[k]) for k in THREAD_ENV if os.environ.get(k, "").isdigit()]
        if capped:
            self.cores = min(capped)
        else:
            try:
                import threadpoolctl
                self.cores = max(i["num_threads"] for i in threadpoolctl.threadpool_info()) or 1
            except Exception:
                self.cores = len(os.sched_getaffinity(0))

    def run(self, n_tok: int) -> float:
        """Seconds for routing, BRIMs (Alg. 3, 5) and the Eq. 1 output of n_tok tokens
        (and, for a training workload, the gradients of x, the weights, the gates and
        the router logits)."""
        from oracle import backward as obackward
        from oracle import brim as obrim
        from oracle import expert as oexpert
        from oracle import routing as orouting
        n_tok = max(1, min(n_tok, self.cfg.T))
        t0 = time.perf_counter()
        ids, gates = orouting.route_topk(self.logits[:n_tok], self.cfg.top_k,
                                         renorm=self.cfg.renorm)
        obrim.Brims(ids, gates, self.L)
        oexpert.layer_output(self.x[:n_tok], ids, gates, self.w)
        if self.dy is not None:
            g = obackward.moe_backward(self.x[:n_tok], ids, gates, self.w["w1"], self.w["w2"],
                                       self.dy[:n_tok])
            obackward.router_grad(self.logits[:n_tok], ids, g["dgates"], renorm=self.cfg.renorm)
        return time.perf_counter() - t0

    def tokens_for(self, seconds: float) -> int:
        """Sample size (<= T) whose run takes about `seconds`, grown from 64 tokens."""
        self.run(16)  # first touch of the weights
        n = 64
        while True:
            dt = self.run(n)
            if n >= self.cfg.T or dt >= 0.5 * seconds:
                break
            n = min(self.cfg.T, max(2 * n, int(n * seconds / max(dt, 1e-3))))
        return n

    def describe(self, n_tok: int, dt: float, runs: int = 1) -> dict:
        return {"value": n_tok * runs / dt, "unit": UNIT, "cores": self.cores, "kind": "oracle",
                "sample": f"first {n_tok} tokens of the {self.cfg.T}-token batch, {runs} run(s): "
                          f"routing, BRIMs (Alg. 3, 5) and the Eq. 1 output"
                          + (" and its backward" if self.dy is not None else "")
                          + f" in fp64, {dt:.1f} s"}


THREAD_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def cpu_baseline_one_thread(cfg, seconds: float = 5.0):
    """The same oracle sample on one host core: a child interpreter whose BLAS and
    OpenMP pools are capped at one thread before numpy loads.  The child sees no
    GPU and draws the batch on the CPU (same shapes and distributions)."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", **{k: "1" for k in THREAD_ENV})
    code = ("import json, sys; sys.path.insert(0, %r); import bench, synth; "
            "cfg = synth.CONFIGS[%r].with_(T=%d); "
            "print(json.dumps(bench.cpu_baseline(cfg, %r)))" % (ROOT, cfg.name, cfg.T, seconds))
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                           timeout=300)
        if r.returncode != 0:
            return {"error": (r.stderr.strip().splitlines() or ["failed"])[-1]}
        return json.loads(r.stdout.strip().splitlines()[-1])
    except (subprocess.TimeoutExpired, OSError, ValueError, IndexError) as e:
        return {"error": f"{type(e).__name__}: {e}"}


def cpu_baseline(cfg, seconds: float = 15.0):
    """About `seconds` of oracle work: runs of up to the whole batch, repeated."""
    o = OracleSample(cfg)
    n = o.tokens_for(seconds)
    total, runs = 0.0, 0
    while total < seconds and total < 30.0:
        total += o.run(n)
        runs += 1
        if total + total / runs > 30.0:
            break
    return o.describe(n, total, runs)


def run_reference(args, cfg, world, rank):
    if rank != 0:
        return
    o = OracleSample(cfg)
    # each step is a bounded sample so that warm-up + timed steps take ~2 minutes
    n = o.tokens_for(120.0 / max(1, args.warmup + args.steps))
    for _ in range(args.warmup):
        o.run(n)
    dt = sum(o.run(n) for _ in range(args.steps))
    v = n * args.steps / dt
    cb = o.describe(n, dt, args.steps)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * cfg.T / v,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": workload_desc(cfg)},
        "cpu_baseline": cb,
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def library_placement(occ, cfg, dev):
    """Algorithm 1 placement the way a user of the library gets it: the profiling
    batch routed on the GPU (plain top-k), its co-activation counts C (Eq. 3) on
    the GPU, then Algorithm 1 on the host, all through the C ABI.  Returns the
    placement and the three steps' times (offline: not part of the timed step)."""
    H = synth.profiling_logits(cfg).to(dev)
    n, Ne, k = H.shape[0], cfg.n_experts, cfg.top_k
    pds = occ.desc_for(cfg.with_(T=n, route_mode="exact"))
    e2v = torch.arange(Ne, dtype=torch.int32, device=dev) // (Ne // cfg.n_vdev)  # masks unused
    ids = torch.empty(n, k, dtype=torch.int32, device=dev)
    gates = torch.empty(n, k, dtype=torch.float32, device=dev)
    vmask = torch.empty(n, dtype=torch.int32, device=dev)
    C = torch.empty(Ne, Ne, dtype=torch.int64, device=dev)
    ws = torch.empty(max(1, occ.workspace_size(pds, occ.WS_PROFILE_COACT, n)), dtype=torch.uint8,
                     device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for _ in range(2):  # the second pass is timed (the first loads the kernels)
        ev[0].record()
        occ.occult_route(pds, H, e2v, ids, gates, vmask)
        ev[1].record()
        occ.occult_profile_coact(pds, ids, n, C, ws)
        ev[2].record()
    torch.cuda.synchronize(dev)
    C_host = C.cpu()
    t0 = time.perf_counter()
    L, _ = occ.occult_place(C_host, cfg.n_vdev)
    place_ms = 1e3 * (time.perf_counter() - t0)
    return L, {"profiling_tokens": n, "route_ms": ev[0].elapsed_time(ev[1]),
               "profile_coact_ms": ev[1].elapsed_time(ev[2]), "place_ms": place_ms}


def run_ours(args, cfg, world, rank, local):
    import combine_top_route_gb300 as occ
    from combine_top_route_gb300 import build

    build.build()
    occ.lib()
    dev = torch.device("cuda", local)
    ds = occ.desc_for(cfg)
    L, offline = library_placement(occ, cfg, dev)
    logits = synth.measured_logits(cfg).to(dev)
    x = synth.hidden_states(cfg, device=dev)
    w = synth.expert_weights(cfg, device=dev)
    train = bool(cfg.backward)
    table = None
    if cfg.route_mode == "similarity_pruned":
        # the similarity table of App. A.3 from the profiling batch (Eq. 8), built
        # by the library; not part of the timed step
        G = torch.zeros(cfg.n_experts, cfg.n_experts, dtype=torch.float64, device=dev)
        H = synth.profiling_logits(cfg).to(dev)
        occ.occult_similarity_accumulate(ds, H, H.shape[0], G)
        table = torch.empty(cfg.n_experts, cfg.n_experts, dtype=torch.float32, device=dev)
        occ.occult_similarity_finish(ds, G, table)
    sharded = cfg.n_src > 1
    src_off = synth.source_offsets(cfg) if sharded else None
    moe = occ.OccultMoE(ds, w, L, device=dev, train=train, sim_table=table, src_off=src_off,
                        merge=args.merge)
    dy = synth.upstream_grad(cfg, device=dev) if train else None
    stream = torch.cuda.current_stream(dev)
    T, k, d, I = cfg.T, cfg.top_k, cfg.d, cfg.inter

    # one step as named C-ABI calls, in Algorithm 2's order (+ the backward)
    if cfg.route_mode == "similarity_pruned":
        route = lambda: occ.occult_route_similarity(  # noqa: E731
            ds, logits, moe.expert_to_vdev, moe.sim_table, moe.ids, moe.gates, moe.vmask,
            moe.routed, stream)
    else:
        route = lambda: occ.occult_route(ds, logits, moe.expert_to_vdev, moe.ids,  # noqa: E731
                                         moe.gates, moe.vmask, stream)
    calls = [
        ("route", route),
        ("build_brim", lambda: occ.occult_build_brim(
            ds, moe.ids, moe.gates, moe.vmask, moe.placement, moe.brim0, moe.seg_off, moe.brim1,
            moe.exp_off, moe.epd_src, moe.epd_gate, moe.counts, moe.brim_ws, stream)),
    ]
    if sharded:
        # the sources' send buffers, then the first all-to-all into the devices'
        # receive buffers
        calls += [
            ("shard_plan", lambda: occ.occult_shard_plan(
                ds, src_off, moe.vmask, moe.brim0, moe.brim0_send, moe.blk_counts, moe.send_off,
                moe.recv_off, stream)),
            ("dispatch", lambda: occ.occult_dispatch(ds, x, moe.brim0_send, moe.vmask,
                                                     moe.x_send, None, stream)),
            ("all_to_all_0", lambda: occ.occult_all_to_all(
                ds, moe.n_src, moe.blk_counts, moe.send_off, moe.recv_off, moe.x_send, moe.x_sfd,
                reverse=False, stream=stream)),
        ]
    else:
        calls.append(("dispatch", lambda: occ.occult_dispatch(ds, x, moe.brim0, moe.vmask,
                                                              moe.x_sfd, moe.sfd_tok, stream)))
    calls.append(("expert_up", lambda: occ.occult_expert_up(
        ds, moe.x_sfd, moe.epd_src, moe.epd_gate, moe.exp_off, moe.placement, moe.w["w1"],
        moe.h_epd, moe.gu_epd, x_epd=moe.x_epd, stream=stream)))
    atomic = moe.merge == "atomic"
    if atomic:
        # shared experts write y; the down-projection adds every EPD row into its
        # token's row of y (fp32 atomics): no separate merge kernel
        if ds.n_shared:
            calls.append(("shared_ffn", lambda: occ.occult_shared_ffn(
                ds, x, moe.w["ws1"], moe.w["ws2"], moe.w.get("w_sg"), moe.h_s, moe.s_gate, moe.y,
                stream)))
        else:
            calls.append(("zero_y", lambda: occ.occult_zero_f32(moe.y, stream)))
        calls.append(("expert_down_merge", lambda: occ.occult_expert_down_merge(
            ds, moe.h_epd, moe.exp_off, moe.placement, moe.w["w2"], moe.epd_src, moe.sfd_tok,
            moe.y, zero_y=False, stream=stream)))
    else:
        calls.append(("expert_down", lambda: occ.occult_expert_down(
            ds, moe.h_epd, moe.exp_off, moe.placement, moe.w["w2"], moe.y_epd, stream)))
        if ds.n_shared:
            calls.append(("shared_ffn", lambda: occ.occult_shared_ffn(
                ds, x, moe.w["ws1"], moe.w["ws2"], moe.w.get("w_sg"), moe.h_s, moe.s_gate,
                moe.y_s, stream)))
    if sharded:
        # stage one, the second all-to-all back to the sources, stage two there
        calls += [
            ("merge_sfd", lambda: occ.occult_merge_sfd(ds, moe.y_epd, moe.brim0, moe.seg_off,
                                                       moe.brim1, moe.exp_off, moe.y_sfd,
                                                       stream)),
            ("all_to_all_1", lambda: occ.occult_all_to_all(
                ds, moe.n_src, moe.blk_counts, moe.send_off, moe.recv_off, moe.y_sfd, moe.y_send,
                reverse=True, stream=stream)),
            ("combine_sfd", lambda: occ.occult_combine_sfd(ds, moe.y_send, moe.brim0_send, moe.y,
                                                           y_shared=moe.y_s, stream=stream)),
        ]
    elif not atomic:
        calls.append(("combine", lambda: occ.occult_combine(ds, moe.y_epd, moe.brim0,
                                                            moe.seg_off, moe.brim1, moe.exp_off,
                                                            moe.y, y_shared=moe.y_s,
                                                            stream=stream)))
    if train and sharded:
        raise SystemExit("the timed training step runs single-source")
    if train:
        calls += [
            # one source: dy straight to the padded EPD rows the backward GEMMs read
            ("dispatch_dy", lambda: occ.occult_dispatch_epd(ds, dy, moe.ids, moe.placement,
                                                            moe.brim0, moe.seg_off, moe.brim1,
                                                            moe.exp_off, moe.dy_epd, stream)),
        ]
        # the expert backward as its four GEMMs (each timed on its own)
        if atomic:
            calls.append(("zero_dx", lambda: occ.occult_zero_f32(moe.dx, stream)))
        calls += [
            ("dgrad_down", lambda: occ.occult_expert_dgrad_down(
                ds, None, moe.epd_src, moe.epd_gate, moe.exp_off, moe.placement,
                moe.w["w2"], moe.gu_epd, moe.dgu_epd, moe.dg_epd, moe.bwd_ws, dy_epd=moe.dy_epd,
                stream=stream)),
            ("dgrad_up", lambda: occ.occult_expert_dgrad_up(
                ds, moe.dgu_epd, moe.epd_src, moe.exp_off, moe.placement, moe.w["w1"],
                moe.dx if atomic else moe.dx_epd, sfd_tok=moe.sfd_tok if atomic else None,
                zero_dx=False, stream=stream)),
            ("wgrad_down", lambda: occ.occult_expert_wgrad_down(
                ds, None, None, moe.exp_off, moe.placement, moe.h_epd, moe.dw2,
                dy_epd=moe.dy_epd, stream=stream)),
            ("wgrad_up", lambda: occ.occult_expert_wgrad_up(
                ds, None, None, moe.exp_off, moe.placement, moe.dgu_epd, moe.dw1,
                x_epd=moe.x_epd, stream=stream)),
        ]
        if not atomic:
            calls.append(("combine_dx", lambda: occ.occult_combine(
                ds, moe.dx_epd, moe.brim0, moe.seg_off, moe.brim1, moe.exp_off, moe.dx,
                stream=stream)))
        calls += [
            ("gate_grad", lambda: occ.occult_gate_grad(ds, moe.ids, moe.placement, moe.brim0,
                                                       moe.seg_off, moe.brim1, moe.exp_off,
                                                       moe.dg_epd, moe.dgates, stream)),
            ("router_grad", lambda: occ.occult_router_grad(ds, logits, moe.routed, moe.dgates,
                                                           moe.dlogits, stream)),
        ]
    names = [c[0] for c in calls]

    def step(ev=None):
        for j, (_, fn) in enumerate(calls):
            if ev is not None:
                ev[j].record(stream)
            fn()
        if ev is not None:
            ev[len(calls)].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # ---- device-timed region: K steps, inputs resident in HBM ----------------
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        start.record(stream)
        for _ in range(args.steps):
            step()
        stop.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    ms_total = max_over_ranks(start.elapsed_time(stop), world)
    ms_step = ms_total / args.steps

    # ---- per-call durations (separate pass with events between calls) ------
    n_prof = min(args.steps, 200)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
           for _ in range(n_prof)]
    torch.cuda.synchronize(dev)
    for i in range(n_prof):
        step(evs[i])
    torch.cuda.synchronize(dev)
    per_call = {c: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(n_prof))
                for j, c in enumerate(names)}
    n_sfd = int(moe.counts[0].item())

    # ---- end to end through the public API with host buffers ----------------
    # Every step copies its inputs from pinned host memory and reads its output
    # back; the copies run on their own streams, double-buffered, so that step
    # i+1's inputs arrive and step i-1's output leaves while step i computes.
    x_h = x.cpu().pin_memory()
    lg_h = logits.cpu().pin_memory()
    y_h = torch.empty(T, d, dtype=torch.float32).pin_memory()
    dy_h = dy.cpu().pin_memory() if train else None
    x_d = [torch.empty_like(x) for _ in range(2)]
    lg_d = [torch.empty_like(logits) for _ in range(2)]
    y_d = [torch.empty(T, d, dtype=torch.float32, device=dev) for _ in range(2)]
    dy_d = [torch.empty_like(dy) for _ in range(2)] if train else None
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_done + ev_out:
        e.record(stream)

    def e2e_step(i):
        b = i & 1
        s_in.wait_event(ev_done[b])          # buffer b's previous step has finished
        with torch.cuda.stream(s_in):
            x_d[b].copy_(x_h, non_blocking=True)
            lg_d[b].copy_(lg_h, non_blocking=True)
            if train:
                dy_d[b].copy_(dy_h, non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])         # y_d[b] has left for the host
        moe.forward(lg_d[b], x_d[b], stream, out=y_d[b])
        if train:
            moe.backward(dy_d[b], stream)
        ev_done[b].record(stream)
        s_out.wait_event(ev_done[b])
        with torch.cuda.stream(s_out):
            y_h.copy_(y_d[b], non_blocking=True)
        ev_out[b].record(s_out)

    n_e2e_warm = max(3, args.warmup // 4)
    for i in range(n_e2e_warm):
        e2e_step(i)
    n_e2e = max(10, args.steps // 4)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    s_in.wait_stream(stream)                 # the first copy starts after the clock does
    for i in range(n_e2e):
        e2e_step(n_e2e_warm + i)
    stream.wait_event(ev_out[(n_e2e_warm + n_e2e - 1) & 1])   # the last output is on the host
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / n_e2e

    hbm, tflops_burst, tflops_sust, peak_src = peaks()
    sustained = ms_total >= SUSTAINED_MS
    tflops = tflops_sust if sustained else tflops_burst
    b = 2  # bytes per bf16 element (x, x_sfd, weights, h); y_epd, y_shared and y are fp32
    n_epd = T * k
    S = cfg.n_shared * cfg.shared_inter
    # algorithmic work per launch: FLOPs and the bytes that must cross HBM once
    # (the training step's up-projection also writes G | U and the padded EPD copy
    # of its gathered x rows for the backward)
    work = {
        "expert_up": (4.0 * d * I * n_epd,
                      cfg.n_experts * 2 * I * d * b + n_sfd * d * b + n_epd * I * b
                      + (n_epd * 2 * I * b + n_epd * d * b if train else 0)),
    }
    if atomic:
        # weights, h, and y written once (read once more when it holds the shared
        # output); the additions themselves stay in L2 (y is 4 bytes x T x d)
        work["expert_down_merge"] = (2.0 * d * I * n_epd, cfg.n_experts * I * d * b
                                     + n_epd * I * b + T * d * 4 * (2 if cfg.n_shared else 1))
    else:
        work["expert_down"] = (2.0 * d * I * n_epd,
                               cfg.n_experts * I * d * b + n_epd * I * b + n_epd * d * 4)
    if S:
        work["shared_ffn"] = (6.0 * d * S * T, 3 * S * d * b + T * d * b + T * S * b + T * d * 4)
    if train:
        # the backward's four GEMMs, twice the forward's FLOPs in all.  Bytes of each:
        #  dgrad_down  W_d, dy's padded EPD rows, G|U read, dG|dU written
        #  dgrad_up    dG|dU, [W_g; W_u], dx written once (merged) or fp32 EPD rows
        #  wgrad_down  the dy rows' EPD copy, h', dW_d written in fp32
        #  wgrad_up    dG|dU, the x rows' EPD copy, dW_g|u written in fp32
        Ne = cfg.n_experts
        work["dgrad_down"] = (2.0 * d * I * n_epd, Ne * d * I * b + n_epd * d * b
                              + 2 * n_epd * 2 * I * b)
        work["dgrad_up"] = (4.0 * d * I * n_epd, n_epd * 2 * I * b + Ne * 2 * I * d * b
                            + (T * d * 4 if atomic else n_epd * d * 4))
        work["wgrad_down"] = (2.0 * d * I * n_epd, n_epd * d * b + n_epd * I * b + Ne * d * I * 4)
        work["wgrad_up"] = (4.0 * d * I * n_epd, n_epd * 2 * I * b + n_epd * d * b
                            + Ne * 2 * I * d * 4)
    ridge = tflops * 1e12 / (hbm * 1e9)  # flop per byte where the two roofs meet
    kernels = {c: {"ms": per_call[c]} for c in names}
    kernels["dispatch"].update({"GB/s": (T * d * b + n_sfd * d * b) / per_call["dispatch"] / 1e6})
    shared_bytes = T * d * 4 if S else 0
    hbm_kernels = ["dispatch"]
    for c, n in (("zero_y", T * d), ("zero_dx", T * d)):
        if c in kernels:
            kernels[c]["GB/s"] = n * 4 / per_call[c] / 1e6
            hbm_kernels.append(c)
    if train:
        kernels["dispatch_dy"]["GB/s"] = (T * d * b + n_epd * d * b) / per_call["dispatch_dy"] / 1e6
        hbm_kernels.append("dispatch_dy")
    if sharded:
        # the exchanges read and write every SFD row once; stage one reads the
        # EPD rows and writes the SFD rows, stage two reads them back
        kernels["all_to_all_0"]["GB/s"] = 2 * n_sfd * d * b / per_call["all_to_all_0"] / 1e6
        kernels["all_to_all_1"]["GB/s"] = 2 * n_sfd * d * 4 / per_call["all_to_all_1"] / 1e6
        kernels["merge_sfd"]["GB/s"] = (n_epd * d * 4 + n_sfd * d * 4) / per_call["merge_sfd"] / 1e6
        kernels["combine_sfd"]["GB/s"] = ((n_sfd * d * 4 + T * d * 4 + shared_bytes)
                                          / per_call["combine_sfd"] / 1e6)
        hbm_kernels += ["all_to_all_0", "all_to_all_1", "merge_sfd", "combine_sfd"]
    elif not atomic:
        kernels["combine"].update({"GB/s": (n_epd * d * 4 + T * d * 4 + shared_bytes)
                                           / per_call["combine"] / 1e6})
        hbm_kernels.append("combine")
    for c, (fl, by) in work.items():
        kernels[c].update({"TFLOP/s": fl / per_call[c] / 1e9, "GB/s": by / per_call[c] / 1e6,
                           "bound": "tensor" if fl / by > ridge else "hbm"})
    dom = max(work, key=lambda c: per_call[c])
    for c in work:
        if kernels[c]["bound"] == "tensor":
            kernels[c]["tensor_frac"] = kernels[c]["TFLOP/s"] / tflops
            kernels[c]["tensor_frac_of_burst"] = kernels[c]["TFLOP/s"] / tflops_burst
    if kernels[dom]["bound"] == "tensor":
        achieved, peak, unit = kernels[dom]["TFLOP/s"], tflops, "TFLOP/s"
        src = (f"{peak_src} bf16 dense {'sustained' if sustained else 'burst'} "
               f"(timed region {ms_total / 1e3:.1f} s"
               + (f"; {kernels[dom]['TFLOP/s'] / tflops_burst:.3f} of the burst figure)"
                  if sustained else ")"))
    else:
        achieved, peak, unit = kernels[dom]["GB/s"], hbm, "GB/s"
        src = f"{peak_src} HBM copy bandwidth"
    roofline = {"bound": kernels[dom]["bound"], "kernel": dom, "achieved": achieved,
                "peak": peak, "unit": unit, "frac": achieved / peak,
                "traffic": (recorded_traffic(cfg.name + ("" if atomic else ":ordered"), dom)
                            if cfg.T == synth.CONFIGS[cfg.name].T else None),
                "peak_source": src}
    for c in hbm_kernels:
        kernels[c]["hbm_frac"] = kernels[c]["GB/s"] / hbm

    w_bytes = (3 * cfg.n_experts * I + 3 * S) * d * b
    result = {
        "metric": METRIC, "value": world * T / (ms_step / 1e3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": workload_desc(cfg),
                   "merge": ("fp32 atomic adds into the token rows (the paper's merging SMM)"
                             if atomic else "fixed-order two-stage merge"),
                   "l2": f"inputs larger than L2 ({w_bytes / 1e6:.0f} MB of expert weights read "
                         "every step)",
                   "parallelism": f"{world} independent replica(s), Nd={cfg.n_vdev} virtual "
                                  "expert-parallel devices each"
                                  + (f", batch split over {cfg.n_src} source shards exchanging "
                                     "row blocks" if sharded else "")},
        "roofline": roofline,
        "kernels": kernels,
        "offline": offline,
        "E[C_T]": n_sfd / T,
        "a2a_bytes_per_direction": n_sfd * d * b,
        "clocks": clk.summary(),
        "gpu_launches": (moe.launches_per_forward + (moe.launches_per_backward if train else 0))
                        * args.steps,
        "e2e": {"value": world * T / (e2e_ms / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": x.numel() * x.element_size() + logits.numel() * 4
                                      + (dy.numel() * dy.element_size() if train else 0),
                "d2h_bytes_per_step": T * d * 4},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(cfg, args.cpu_seconds)
        result["cpu_baseline"]["one_thread"] = cpu_baseline_one_thread(cfg)
    if rank == 0:
        print(json.dumps(result), flush=True)


def main():
    args = parse()
    world, rank, local = dist_setup(args.gpus)
    cfg = synth.CONFIGS[args.config]
    if args.tokens is not None:
        cfg = cfg.with_(T=args.tokens)
    if args.impl == "reference":
        run_reference(args, cfg, world, rank)
    else:
        run_ours(args, cfg, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
