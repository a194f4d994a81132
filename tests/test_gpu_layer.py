"""GPU parity of every step of the Occult layer against the CPU oracle, through
the C ABI.  Integer and index outputs are compared bit for bit, floating-point
outputs at the stated tolerances.  No oracle input or expected value comes from
the CUDA path: the GPU is fed the oracle's own routing where a step needs it.
"""
import numpy as np
import pytest
import torch

import synth
from layer_cases import (alg1_placement, assert_close_layer, h_bound, make_case, oracle_brims,
                         reference_output, sfd_bound)
from oracle import brim as obrim
from oracle import coact as ocoact
from oracle import expert as oexpert
from oracle import placement as oplace
from oracle import routing as orouting

pytestmark = pytest.mark.gpu

# relative tolerance of the fp32 gates: exp (2 ulp), argument rounding, a 6-level
# sum tree and the division stay below ~25 ulp (2^-24 each) ~ 1.5e-6
GATE_RTOL = 2e-6

CFG = dict(synth.CONFIGS)
ALL = ["tiny_f32", "olmoe_fwd", "qwen_prefill", "deepseek_decode", "deepseek_decode_limited",
       "olmoe_train"]
# shapes that exercise edges: ragged T, one token, one device, one expert per
# device, k = 1, k = Nd
EDGE = {
    "ragged_1000": CFG["olmoe_fwd"].with_(name="ragged_1000", T=1000),
    "one_token": CFG["olmoe_fwd"].with_(name="one_token", T=1),
    "t33_nd1": CFG["tiny_f32"].with_(name="t33_nd1", T=33, n_vdev=1),
    "nloc1": CFG["tiny_f32"].with_(name="nloc1", T=77, n_vdev=8),
    "k1_bf16": CFG["olmoe_fwd"].with_(name="k1_bf16", T=300, top_k=1, d=256, inter=128),
    "k_eq_nd": CFG["olmoe_fwd"].with_(name="k_eq_nd", T=513, d=512, inter=192, n_vdev=8),
    # >= 256 rows an expert on average: the GEMMs run on CTA pairs, with ragged
    # segments (pair units whose second tile is partial or empty)
    "pair_ragged": CFG["olmoe_fwd"].with_(name="pair_ragged", T=2500, d=512, inter=320),
    # the largest layers the ABI takes: 256 experts, 32 virtual devices, k = 16; and
    # 128 experts on 16 devices with k = 12
    "ne256_nd32_k16": CFG["olmoe_fwd"].with_(name="ne256_nd32_k16", T=700, d=256, inter=128,
                                             n_experts=256, top_k=16, n_vdev=32, n_clusters=16,
                                             experts_per_cluster=24, prof_tokens=4096),
    "ne128_nd16_k12": CFG["olmoe_fwd"].with_(name="ne128_nd16_k12", T=513, d=512, inter=192,
                                             n_experts=128, top_k=12, n_vdev=16, n_clusters=16,
                                             experts_per_cluster=16, prof_tokens=4096),
}


@pytest.fixture(scope="session")
def occ():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_top_route_gb300 import build
    build.build()
    import combine_top_route_gb300 as occ
    occ.lib()
    return occ


def cuda(a, dtype=None):
    t = torch.as_tensor(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def i32(a):
    return cuda(np.asarray(a, dtype=np.int64).astype(np.int32))


def vmask_bits(ids, e2v):
    act = orouting.token_devices(ids, e2v, int(e2v.max()) + 1)
    bits = np.zeros(ids.shape[0], dtype=np.int64)
    for d in range(act.shape[1]):
        bits |= act[:, d].astype(np.int64) << d
    return bits.astype(np.uint32).view(np.int32)


def sample_tokens(T, n=128, seed=0):
    if T <= n:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(16, T - 16), size=n - 32, replace=False)
    return np.unique(np.concatenate([np.arange(16), mid, np.arange(T - 16, T)]))


# --------------------------------------------------------------------------- route
@pytest.mark.parametrize("name", ALL + list(EDGE))
def test_route(occ, name):
    cfg = CFG.get(name) or EDGE[name]
    case = make_case(cfg, device="cpu", tensors=False)
    ids_o, gates_o, margin = case.oracle_route()
    ds = occ.desc_for(cfg)
    T, k = cfg.T, cfg.top_k
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    gates = torch.empty(T, k, dtype=torch.float32, device="cuda")
    vmask = torch.empty(T, dtype=torch.int32, device="cuda")
    occ.occult_route(ds, case.logits.cuda(), i32(case.e2v), ids, gates, vmask)
    torch.cuda.synchronize()
    ids_g, gates_g, vm_g = ids.cpu().numpy(), gates.cpu().numpy(), vmask.cpu().numpy()
    sure = margin > 1e-5   # device-limited choices that rounding cannot flip
    assert (ids_g[sure] == ids_o[sure]).all()
    np.testing.assert_allclose(gates_g[sure], gates_o[sure], rtol=GATE_RTOL, atol=0)
    assert (vm_g[sure] == vmask_bits(ids_o, case.e2v)[sure]).all()
    # any token whose device choice hangs on rounding must still be a valid choice
    for t in np.nonzero(~sure)[0]:
        devs = {int(case.e2v[e]) for e in ids_g[t]}
        assert len(devs) <= cfg.limit_devices and len(set(ids_g[t])) == k
    if cfg.route_mode == "device_limited":
        ct = np.array([bin(v & 0xffffffff).count("1") for v in vm_g.astype(np.int64)])
        assert ct.max() <= cfg.limit_devices


# --------------------------------------------------------------------------- BRIM
def run_brim(occ, case, ids_o, gates_o):
    cfg = case.cfg
    T, k, Ne, Nd = cfg.T, cfg.top_k, cfg.n_experts, cfg.n_vdev
    ds = occ.desc_for(cfg)
    out = dict(brim0=torch.full((Nd, T), -7, dtype=torch.int32, device="cuda"),
               seg_off=torch.empty(Nd + 1, dtype=torch.int32, device="cuda"),
               brim1=torch.full((Ne, T), -7, dtype=torch.int32, device="cuda"),
               exp_off=torch.empty(Ne + 1, dtype=torch.int32, device="cuda"),
               epd_src=torch.full((T * k,), -7, dtype=torch.int32, device="cuda"),
               epd_gate=torch.empty(T * k, dtype=torch.float32, device="cuda"),
               counts=torch.empty(4, dtype=torch.int32, device="cuda"),
               ws=torch.empty(max(1, occ.workspace_size(ds, occ.WS_BUILD_BRIM)),
                              dtype=torch.uint8, device="cuda"))
    occ.occult_build_brim(ds, i32(ids_o), cuda(gates_o.astype(np.float32)),
                          cuda(vmask_bits(ids_o, case.e2v)), i32(case.placement), **out)
    torch.cuda.synchronize()
    out.pop("ws")
    return {n: v.cpu().numpy() for n, v in out.items()}


@pytest.mark.parametrize("name", ALL + list(EDGE))
def test_brim_bit_exact(occ, name):
    cfg = CFG.get(name) or EDGE[name]
    case = make_case(cfg, device="cpu", tensors=False)
    ids_o, gates_o, _ = case.oracle_route()
    g32 = gates_o.astype(np.float32)
    b = oracle_brims(case, ids_o, g32)
    got = run_brim(occ, case, ids_o, g32)
    assert (got["brim0"] == b.brim0).all()
    assert (got["seg_off"] == b.seg_off).all()
    assert (got["exp_off"] == b.exp_off).all()
    assert (got["epd_src"] == b.epd_src).all()
    assert (got["epd_gate"] == b.epd_gate.astype(np.float32)).all()
    n_loc = cfg.n_loc
    for d in range(cfg.n_vdev):
        n_d = int(b.seg_off[d + 1] - b.seg_off[d])
        assert (got["brim1"][d * n_loc:(d + 1) * n_loc, :n_d] == b.brim1[d]).all()
    ct = b.ct
    assert got["counts"][:3].tolist() == [b.n_sfd, cfg.T * cfg.top_k, int(ct.max()) if ct.size else 0]
    lo, hi = ocoact.ct_bounds(cfg.top_k, cfg.n_experts, cfg.n_vdev)
    assert cfg.T == 0 or (lo <= ct.min() and ct.max() <= hi)


def test_brim_skewed_routing(occ):
    """Every token routes to the same k experts: one long segment per expert."""
    cfg = CFG["olmoe_fwd"].with_(T=2048)
    lg = torch.zeros(cfg.T, cfg.n_experts)
    lg[:, [3, 17, 40, 41, 42, 50, 60, 63]] = 5.0
    case = make_case(cfg, device="cpu", logits=lg, tensors=False)
    ids_o, gates_o, _ = case.oracle_route()
    g32 = gates_o.astype(np.float32)
    b = oracle_brims(case, ids_o, g32)
    got = run_brim(occ, case, ids_o, g32)
    assert (got["brim0"] == b.brim0).all() and (got["epd_src"] == b.epd_src).all()
    assert (got["exp_off"] == b.exp_off).all()


# --------------------------------------------------------------------------- dispatch
@pytest.mark.parametrize("name", ["tiny_f32", "olmoe_fwd", "qwen_prefill", "ragged_1000",
                                  "one_token"])
def test_dispatch_bit_exact(occ, name):
    cfg = CFG.get(name) or EDGE[name]
    case = make_case(cfg)
    ids_o, gates_o, _ = case.oracle_route()
    b = oracle_brims(case, ids_o, gates_o)
    ds = occ.desc_for(cfg)
    n_max = cfg.T * min(cfg.top_k, cfg.n_vdev)
    x_sfd = torch.zeros(n_max, cfg.d, dtype=cfg.torch_dtype, device="cuda")
    sfd_tok = torch.full((n_max,), -1, dtype=torch.int32, device="cuda")
    occ.occult_dispatch(ds, case.x, i32(b.brim0), cuda(vmask_bits(ids_o, case.e2v)), x_sfd, sfd_tok)
    torch.cuda.synchronize()
    want = obrim.dispatch(case.host("x"), b.brim0)
    assert (x_sfd[:b.n_sfd].float().cpu().numpy() == want).all()
    assert (sfd_tok[:b.n_sfd].cpu().numpy() == np.concatenate(b.row_tokens)).all()


# --------------------------------------------------------------------------- expert GEMMs
def epd_sample(b, n=256, seed=1):
    """EPD rows to check: every row of the first, a middle and the last slot, plus random rows."""
    rng = np.random.default_rng(seed)
    Ne = len(b.exp_off) - 1
    rows = [np.arange(b.exp_off[s], b.exp_off[s + 1]) for s in (0, Ne // 2, Ne - 1)]
    rows.append(rng.integers(0, max(b.n_epd, 1), size=min(n, b.n_epd)))
    return np.unique(np.concatenate(rows)).astype(np.int64)


@pytest.mark.parametrize("name", ALL + ["ragged_1000", "k1_bf16", "k_eq_nd", "nloc1",
                                  "pair_ragged"])
def test_expert_up(occ, name):
    cfg = CFG.get(name) or EDGE[name]
    case = make_case(cfg)
    ids_o, gates_o, _ = case.oracle_route()
    g32 = gates_o.astype(np.float32)
    b = oracle_brims(case, ids_o, g32)
    ds = occ.desc_for(cfg)
    x = case.host("x")
    n_max = cfg.T * min(cfg.top_k, cfg.n_vdev)
    x_sfd = np.zeros((n_max, cfg.d), np.float32)
    x_sfd[:b.n_sfd] = obrim.dispatch(x, b.brim0)
    h = torch.full((cfg.T * cfg.top_k, cfg.inter), float("nan"), dtype=cfg.torch_dtype,
                   device="cuda")
    occ.occult_expert_up(ds, cuda(x_sfd, cfg.torch_dtype), i32(b.epd_src),
                         cuda(b.epd_gate.astype(np.float32)),
                         i32(b.exp_off), i32(case.placement.reshape(-1)),
                         case.weights["w1"], h)
    torch.cuda.synchronize()
    rows = epd_sample(b)
    w1 = case.host("w1")
    I = cfg.inter
    got = h[torch.as_tensor(rows, device="cuda")].float().cpu().numpy()
    for i, r in enumerate(rows):
        e = b.epd_exp[r]
        a = x[b.epd_tok[r]].astype(np.float64)
        ref = b.epd_gate[r] * oexpert.silu(w1[e, :I] @ a) * (w1[e, I:] @ a)
        bound = h_bound(a, w1[e, :I], w1[e, I:], float(b.epd_gate[r]), ref, cfg.dtype)
        err = np.abs(got[i] - ref)
        assert (err <= bound).all(), (
            f"h_epd row {r}: worst excess {float(np.max(err - bound)):.3e}")
    assert np.isfinite(h.float().cpu().numpy()).all(), "an EPD row was left unwritten"


@pytest.mark.parametrize("name", ALL + ["ragged_1000", "k1_bf16", "nloc1", "pair_ragged"])
def test_expert_down(occ, name):
    cfg = CFG.get(name) or EDGE[name]
    case = make_case(cfg)
    ids_o, gates_o, _ = case.oracle_route()
    b = oracle_brims(case, ids_o, gates_o)
    ds = occ.desc_for(cfg)
    g = torch.Generator().manual_seed(11)
    h = torch.randn(cfg.T * cfg.top_k, cfg.inter, generator=g).to(cfg.torch_dtype)
    y = torch.full((cfg.T * cfg.top_k, cfg.d), float("nan"), dtype=torch.float32, device="cuda")
    occ.occult_expert_down(ds, h.cuda(), i32(b.exp_off), i32(case.placement.reshape(-1)),
                           case.weights["w2"], y)
    torch.cuda.synchronize()
    rows = epd_sample(b)
    w2 = case.host("w2")
    hh = h.float().numpy().astype(np.float64)
    ref = np.stack([w2[b.epd_exp[r]] @ hh[r] for r in rows]) if rows.size else np.zeros((0, cfg.d))
    got = y[torch.as_tensor(rows, device="cuda")].float().cpu().numpy()
    assert_close_layer(got, ref, cfg.dtype, "y_epd")
    assert np.isfinite(y.float().cpu().numpy()).all(), "an EPD row was left unwritten"


def test_unaligned_output_is_refused(occ):
    """A bf16 layer's GEMM output must start on a 16-byte boundary (its epilogues
    store 16-byte vectors): one that does not is refused before any launch and
    the buffer is left as it was."""
    cfg = CFG["olmoe_fwd"].with_(name="unaligned", T=64)
    case = make_case(cfg)
    ids_o, gates_o, _ = case.oracle_route()
    b = oracle_brims(case, ids_o, gates_o)
    ds = occ.desc_for(cfg)
    h = torch.zeros(cfg.T * cfg.top_k, cfg.inter, dtype=cfg.torch_dtype, device="cuda")
    buf = torch.full((cfg.T * cfg.top_k * cfg.d + 1,), 7.0, dtype=torch.float32, device="cuda")
    y = buf[1:].view(cfg.T * cfg.top_k, cfg.d)          # 4 bytes past a 16-byte boundary
    with pytest.raises(occ.OccultError) as e:
        occ.occult_expert_down(ds, h, i32(b.exp_off), i32(case.placement.reshape(-1)),
                               case.weights["w2"], y)
    assert e.value.code == occ.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert (buf == 7.0).all()
    assert occ.device_error() == 0


# --------------------------------------------------------------------------- shared experts
@pytest.mark.parametrize("name", ["qwen_prefill", "deepseek_decode"])
def test_shared_ffn(occ, name):
    cfg = CFG[name].with_(T=1000)
    case = make_case(cfg)
    ds = occ.desc_for(cfg)
    S = cfg.n_shared * cfg.shared_inter
    h_s = torch.empty(cfg.T, S, dtype=cfg.torch_dtype, device="cuda")
    y_s = torch.empty(cfg.T, cfg.d, dtype=torch.float32, device="cuda")
    s_gate = torch.empty(cfg.T, dtype=torch.float32, device="cuda")
    occ.occult_shared_ffn(ds, case.x, case.weights["ws1"], case.weights["ws2"],
                          case.weights.get("w_sg"), h_s, s_gate, y_s)
    torch.cuda.synchronize()
    toks = sample_tokens(cfg.T)
    ref = oexpert.shared_experts(case.host("x"), case.host("ws1"), case.host("ws2"),
                                 case.host("w_sg") if cfg.shared_gate else None, toks)
    assert_close_layer(y_s.float().cpu().numpy()[toks], ref, cfg.dtype, "y_shared")
    if cfg.shared_gate:
        sg = oexpert.shared_gate(case.host("x")[toks], case.host("w_sg"))
        np.testing.assert_allclose(s_gate.cpu().numpy()[toks], sg, rtol=1e-5, atol=1e-6)


# --------------------------------------------------------------------------- whole layer
def run_layer(occ, case, materialize=False, merge=None):
    from combine_top_route_gb300 import OccultMoE
    ds = occ.desc_for(case.cfg)
    moe = OccultMoE(ds, case.weights, torch.as_tensor(case.placement), materialize_sfd=materialize,
                    merge=merge)
    y = moe.forward(case.logits.cuda(), case.x)
    torch.cuda.synchronize()
    return moe, y


@pytest.mark.parametrize("name", ALL + list(EDGE))
def test_layer_matches_eq1(occ, name):
    """Occult without pruning reaches the standard top-k MoE output (Eq. 1); the
    merge adds each token's rows with fp32 atomics (the default)."""
    cfg = CFG.get(name) or EDGE[name]
    case = make_case(cfg)
    moe, y = run_layer(occ, case)
    assert moe.merge == "atomic"
    ids_o, gates_o, margin = case.oracle_route()
    toks = sample_tokens(cfg.T, 64 if cfg.T > 4096 else 128)
    toks = toks[margin[toks] > 1e-5]
    ref = reference_output(case, toks, ids_o, gates_o)
    assert_close_layer(y.float().cpu().numpy()[toks], ref, cfg.dtype)
    assert occ.device_error() == 0


@pytest.mark.parametrize("name", ["tiny_f32", "k_eq_nd"])
def test_materialised_sfd_matches_staged_oracle(occ, name):
    """Stage one written out (second all-to-all's send buffer) equals Alg. 8's SFD sums."""
    cfg = CFG.get(name) or EDGE[name]
    case = make_case(cfg)
    moe, y = run_layer(occ, case, materialize=True)
    ids_o, gates_o, _ = case.oracle_route()
    y_ref, stages = obrim.occult_forward_staged(case.host("x"), ids_o, gates_o, case.placement,
                                                case.host("w1"), case.host("w2"))
    n_sfd = stages["y_sfd"].shape[0]
    got = moe.y_sfd[:n_sfd].float().cpu().numpy()
    b = oracle_brims(case, ids_o, gates_o)
    w2 = case.host("w2")
    h_abs = np.abs(stages["h_epd"])
    rows_of = [[] for _ in range(n_sfd)]
    for r in range(b.n_epd):
        rows_of[b.epd_src[r]].append((int(b.epd_exp[r]), h_abs[r]))
    for v in range(n_sfd):
        bound = sfd_bound(w2, rows_of[v], cfg.dtype)
        err = np.abs(got[v] - stages["y_sfd"][v])
        assert (err <= bound).all(), f"y_sfd row {v}: worst excess {float(np.max(err - bound)):.3e}"
    assert_close_layer(y.float().cpu().numpy(), y_ref, cfg.dtype)


def test_placement_leaves_output_unchanged(occ):
    cfg = CFG["olmoe_fwd"].with_(T=1024)
    y = {}
    for mode in ("alg1", "trivial", "random"):
        case = make_case(cfg, placement=mode)
        _, out = run_layer(occ, case)
        y[mode] = out.float().cpu().numpy()
    # same seeds on the same device: every case holds the same x and weights
    ref = reference_output(case, np.arange(64))
    for mode, out in y.items():
        assert_close_layer(out[:64], ref, "bf16", f"y[{mode}]")


def test_deterministic_bitwise(occ):
    """The ordered merge is bit-reproducible."""
    case = make_case(CFG["olmoe_fwd"].with_(T=2048))
    _, y1 = run_layer(occ, case, merge="ordered")
    y1 = y1.clone()
    _, y2 = run_layer(occ, case, merge="ordered")
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("name", ["tiny_f32", "olmoe_fwd", "qwen_prefill", "deepseek_decode",
                                  "pair_ragged", "one_token"])
def test_atomic_merge_equals_ordered_merge(occ, name):
    """Both merges sum the same fp32 rows (and the shared output); they differ only
    by the order of the additions: |diff| <= 2 (k + 2) 2^-24 sum|terms| per element.
    The ordered merge also meets Eq. 1 on its own."""
    cfg = CFG.get(name) or EDGE[name]
    case = make_case(cfg)
    moe_o, y_o = run_layer(occ, case, merge="ordered")
    y_o = y_o.clone()
    moe_a, y_a = run_layer(occ, case, merge="atomic")
    ids_o, gates_o, margin = case.oracle_route()
    b = oracle_brims(case, ids_o, gates_o)
    # sum of |rows| of every token, from the ordered run's fp32 EPD rows
    y_epd = moe_o.y_epd[:b.n_epd].cpu().numpy().astype(np.float64)
    S = np.zeros((cfg.T, cfg.d))
    np.add.at(S, b.epd_tok, np.abs(y_epd))
    if cfg.n_shared:
        S += np.abs(moe_o.y_s.cpu().numpy())
    bound = 2 * (cfg.top_k + 2) * 2.0 ** -24 * S + 1e-30
    err = np.abs(y_a.cpu().numpy().astype(np.float64) - y_o.cpu().numpy())
    assert (err <= bound).all(), f"worst excess {float(np.max(err - bound)):.3e}"
    toks = sample_tokens(cfg.T, 64)
    toks = toks[margin[toks] > 1e-5]
    assert_close_layer(y_o.cpu().numpy()[toks], reference_output(case, toks, ids_o, gates_o),
                       cfg.dtype)


def test_empty_batch(occ):
    cfg = CFG["olmoe_fwd"].with_(T=0)
    ds = occ.desc_for(cfg)
    z = torch.empty(0, device="cuda")
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    counts = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    seg = torch.full((cfg.n_vdev + 1,), -1, dtype=torch.int32, device="cuda")
    eo = torch.full((cfg.n_experts + 1,), -1, dtype=torch.int32, device="cuda")
    L = i32(alg1_placement(cfg).reshape(-1))
    occ.occult_route(ds, z, L, e, z, e)
    occ.occult_build_brim(ds, e, z, e, L, e, seg, e, eo, e, z, counts, None)
    torch.cuda.synchronize()
    assert counts[:3].tolist() == [0, 0, 0]
    assert (seg == 0).all() and (eo == 0).all()


# --------------------------------------------------------------------------- profiling
@pytest.mark.parametrize("name", ["tiny_f32", "olmoe_fwd", "qwen_prefill", "olmoe_train",
                                  "ne256_nd32_k16", "ne128_nd16_k12"])
def test_profile_coact_bit_exact(occ, name):
    cfg = CFG.get(name) or EDGE[name]
    lg = synth.profiling_logits(cfg).numpy()
    ids, _ = orouting.route_topk(lg, cfg.top_k)
    L = alg1_placement(cfg)
    e2v = oplace.expert_to_vdev(L)
    ds = occ.desc_for(cfg)
    n = ids.shape[0]
    C = torch.empty(cfg.n_experts, cfg.n_experts, dtype=torch.int64, device="cuda")
    P = torch.empty(cfg.n_experts, cfg.n_experts, dtype=torch.float32, device="cuda")
    hist = torch.empty(min(cfg.top_k, cfg.n_vdev) + 1, dtype=torch.int64, device="cuda")
    ws = torch.empty(occ.workspace_size(ds, occ.WS_PROFILE_COACT, n), dtype=torch.uint8,
                     device="cuda")
    occ.occult_profile_coact(ds, i32(ids), n, C, ws, P=P, vmask=cuda(vmask_bits(ids, e2v)),
                             ct_hist=hist)
    torch.cuda.synchronize()
    C_o = ocoact.coactivation(ids, cfg.n_experts)
    assert (C.cpu().numpy() == C_o).all()
    np.testing.assert_allclose(P.cpu().numpy(), ocoact.normalise(C_o), rtol=2 ** -23, atol=0)
    ct = ocoact.replicas_per_token(ids, e2v)
    assert (hist.cpu().numpy() == ocoact.ct_histogram(ct, min(cfg.top_k, cfg.n_vdev))).all()
    # the host placement of the library reproduces the oracle's Algorithm 1
    Lg, e2v_g = occ.occult_place(C.cpu(), cfg.n_vdev)
    assert (Lg.numpy() == oplace.place(C_o, cfg.n_vdev)).all()
