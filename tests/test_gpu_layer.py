"""GPU parity of every step of the Occult layer against the CPU oracle, through
the C ABI.  Integer and index outputs are compared bit for bit, floating-point
outputs at the stated tolerances.  No oracle input or expected value comes from
the CUDA path: the GPU is fed the oracle's own routing where a step needs it.
"""
import numpy as np
import pytest
import torch

import synth
from layer_cases import (F32_EPS, abs_contract, alg1_placement, assert_close_layer, h_bound,
                         make_case, oracle_brims, reference_output, scatter_add_rows, sfd_bound)
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


# --------------------------------------------------------------------------- route
def assert_valid_device_limited(z, ids_g, gates_g, vm_g, e2v, cfg, tol=1e-5):
    """A device-limited choice that rounding may flip (two device masses within
    ``tol`` of each other) is valid when some set of ``limit_devices`` devices
    (i) holds every device whose mass clearly exceeds the cut and otherwise only
    devices within ``tol`` of it, (ii) has the GPU's ids as its top k experts by
    logit (larger first, ties to the lower id), and (iii) the gates are those
    experts' softmax probabilities renormalised over the k; vmask is the ids'
    devices."""
    import itertools
    Nd, n_keep, k = cfg.n_vdev, cfg.limit_devices, cfg.top_k
    mass = orouting.device_mass(z[None], e2v, Nd)[0].astype(np.float64)
    cut = np.sort(mass)[::-1][n_keep - 1]
    must = [d for d in range(Nd) if mass[d] > cut * (1 + tol)]
    near = [d for d in range(Nd) if d not in must and mass[d] >= cut * (1 - tol)]
    assert len(must) <= n_keep <= len(must) + len(near)
    zz = z.astype(np.float32)
    ok = False
    for extra in itertools.combinations(near, n_keep - len(must)):
        kept = set(must) | set(extra)
        cand = [e for e in range(cfg.n_experts) if int(e2v[e]) in kept]
        order = sorted(cand, key=lambda e: (-float(zz[e]), e))[:k]
        if [int(e) for e in ids_g] == order:
            ok = True
            break
    assert ok, f"ids {ids_g.tolist()} are not the top {k} of any admissible device set"
    ez = np.exp(z[ids_g].astype(np.float64) - float(np.max(z)))
    np.testing.assert_allclose(gates_g, ez / ez.sum(), rtol=GATE_RTOL, atol=0)
    bits = 0
    for e in ids_g:
        bits |= 1 << int(e2v[e])
    assert (int(vm_g) & 0xffffffff) == bits


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
    lg = case.logits.numpy()
    for t in np.nonzero(~sure)[0]:
        assert_valid_device_limited(lg[t], ids_g[t], gates_g[t], vm_g[t], case.e2v, cfg)
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
    check_h_all_rows(h.float().cpu().numpy(), b, x, case.host("w1"), cfg)


def check_h_all_rows(h, b, x, w1, cfg):
    """Every EPD row of h' against Alg. 6-7 (g silu(W_g a) * (W_u a), a the row's
    token input), within the per-element bound of its arithmetic; one expert's
    segment at a time."""
    I = cfg.inter
    assert np.isfinite(h).all(), "an EPD row was left unwritten"
    worst = 0.0
    for s in range(len(b.exp_off) - 1):
        r0, r1 = int(b.exp_off[s]), int(b.exp_off[s + 1])
        if r1 == r0:
            continue
        e = int(b.epd_exp[r0])
        assert (b.epd_exp[r0:r1] == e).all()
        a = x[b.epd_tok[r0:r1]].astype(np.float64)
        g = b.epd_gate[r0:r1].astype(np.float64)
        G = a @ w1[e, :I].T.astype(np.float64)
        U = a @ w1[e, I:].T.astype(np.float64)
        ref = g[:, None] * oexpert.silu(G) * U
        bound = h_bound(a, w1[e, :I], w1[e, I:], g, ref, cfg.dtype)
        err = np.abs(h[r0:r1] - ref)
        assert (err <= bound).all(), (
            f"h_epd rows of slot {s} (expert {e}): worst excess {float(np.max(err - bound)):.3e}")
        worst = max(worst, float(np.max(err / (bound + 1e-300))))
    print(f"h_epd: worst diff/bound {worst:.3f}")


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
    check_y_epd_all_rows(y.float().cpu().numpy(), h.float().numpy(), b, case.host("w2"), cfg)


def check_y_epd_all_rows(y, h, b, w2, cfg):
    """Every EPD row of the second linear layer (Alg. 8 before the merge) against
    W_d h' in fp64, at the layer tolerance."""
    assert np.isfinite(y[:b.n_epd]).all(), "an EPD row was left unwritten"
    ref = np.zeros((b.n_epd, cfg.d))
    for s in range(len(b.exp_off) - 1):
        r0, r1 = int(b.exp_off[s]), int(b.exp_off[s + 1])
        if r1 > r0:
            e = int(b.epd_exp[r0])
            ref[r0:r1] = h[r0:r1].astype(np.float64) @ w2[e].T.astype(np.float64)
    assert_close_layer(y[:b.n_epd], ref, cfg.dtype, "y_epd")


@pytest.mark.parametrize("name", ["tiny_f32", "olmoe_fwd", "qwen_prefill", "deepseek_decode",
                                  "pair_ragged", "k1_bf16"])
def test_expert_ffn(occ, name):
    """occult_expert_ffn (Alg. 6-8 without the merge): every EPD row of h' within
    its derived bound, and every row of y_epd against the oracle's fp64 expert
    output g W_d (silu(W_g a) * (W_u a)) at the layer tolerance."""
    cfg = CFG.get(name) or EDGE[name]
    case = make_case(cfg)
    ids_o, gates_o, _ = case.oracle_route()
    b = oracle_brims(case, ids_o, gates_o.astype(np.float32))
    ds = occ.desc_for(cfg)
    x, w1, w2 = case.host("x"), case.host("w1"), case.host("w2")
    n_max = cfg.T * min(cfg.top_k, cfg.n_vdev)
    x_sfd = np.zeros((n_max, cfg.d), np.float32)
    x_sfd[:b.n_sfd] = obrim.dispatch(x, b.brim0)
    n_epd = cfg.T * cfg.top_k
    h = torch.full((n_epd, cfg.inter), float("nan"), dtype=cfg.torch_dtype, device="cuda")
    y = torch.full((n_epd, cfg.d), float("nan"), dtype=torch.float32, device="cuda")
    occ.occult_expert_ffn(ds, cuda(x_sfd, cfg.torch_dtype), i32(b.epd_src),
                          cuda(b.epd_gate.astype(np.float32)), i32(b.exp_off),
                          i32(case.placement.reshape(-1)), case.weights["w1"],
                          case.weights["w2"], h, y)
    torch.cuda.synchronize()
    check_h_all_rows(h.float().cpu().numpy(), b, x, w1, cfg)
    # y_epd = W_d h' from the oracle's fp64 h'; the GPU reads its own h' (within
    # h_bound of the oracle's) and accumulates I products in fp32:
    #   |dy| <= |W_d| h_b + 2 I 2^-24 |W_d| (|h'| + h_b)
    # (one EPD row is heavy-tailed like h', so the 2e-2 rms bar of the layer
    # output, a sum of k rows, does not apply to it)
    I = cfg.inter
    got = y.cpu().numpy()
    assert np.isfinite(got).all(), "an EPD row was left unwritten"
    worst = 0.0
    for s in range(len(b.exp_off) - 1):
        r0, r1 = int(b.exp_off[s]), int(b.exp_off[s + 1])
        if r1 == r0:
            continue
        e = int(b.epd_exp[r0])
        a = x[b.epd_tok[r0:r1]].astype(np.float64)
        g = b.epd_gate[r0:r1].astype(np.float64)
        hh = g[:, None] * oexpert.silu(a @ w1[e, :I].T) * (a @ w1[e, I:].T)
        h_b = h_bound(a, w1[e, :I], w1[e, I:], g, hh, cfg.dtype)
        ref = hh @ w2[e].T.astype(np.float64)
        wd_abs = np.abs(w2[e]).T
        bound = (abs_contract(h_b, wd_abs)
                 + 2 * I * F32_EPS * abs_contract(np.abs(hh) + h_b, wd_abs) + 1e-30)
        err = np.abs(got[r0:r1] - ref)
        assert (err <= bound).all(), (
            f"y_epd rows of slot {s} (expert {e}): worst excess {float(np.max(err - bound)):.3e}")
        worst = max(worst, float(np.max(err / bound)))
    print(f"y_epd: worst diff/bound {worst:.3f}")
    assert occ.device_error() == 0


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
    ref = oexpert.shared_experts(case.host("x"), case.host("ws1"), case.host("ws2"),
                                 case.host("w_sg") if cfg.shared_gate else None)
    assert_close_layer(y_s.float().cpu().numpy(), ref, cfg.dtype, "y_shared")
    if cfg.shared_gate:
        sg = oexpert.shared_gate(case.host("x"), case.host("w_sg"))
        np.testing.assert_allclose(s_gate.cpu().numpy(), sg, rtol=1e-5, atol=1e-6)


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
    # every token whose routing rounding cannot flip (the others are checked for
    # validity in test_route); the bar is taken over the whole output
    toks = np.nonzero(margin > 1e-5)[0]
    ref = reference_output_chunked(case, toks, ids_o, gates_o)
    assert_close_layer(y.float().cpu().numpy()[toks], ref, cfg.dtype)
    assert occ.device_error() == 0


def reference_output_chunked(case, toks, ids, gates, chunk=4096):
    """The oracle's Eq. 1 output of the listed tokens, computed a chunk of tokens
    at a time (the oracle holds k rows of d per token while it sums)."""
    out = np.empty((len(toks), case.cfg.d))
    for i in range(0, len(toks), chunk):
        out[i:i + chunk] = reference_output(case, toks[i:i + chunk], ids, gates)
    return out


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
    ref = reference_output(case, np.arange(cfg.T))
    for mode, out in y.items():
        assert_close_layer(out, ref, "bf16", f"y[{mode}]")


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
    scatter_add_rows(S, b.epd_tok, np.abs(y_epd))
    if cfg.n_shared:
        S += np.abs(moe_o.y_s.cpu().numpy())
    bound = 2 * (cfg.top_k + 2) * 2.0 ** -24 * S + 1e-30
    err = np.abs(y_a.cpu().numpy().astype(np.float64) - y_o.cpu().numpy())
    assert (err <= bound).all(), f"worst excess {float(np.max(err - bound)):.3e}"
    toks = np.nonzero(margin > 1e-5)[0]
    assert_close_layer(y_o.cpu().numpy()[toks],
                       reference_output_chunked(case, toks, ids_o, gates_o), cfg.dtype)


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
