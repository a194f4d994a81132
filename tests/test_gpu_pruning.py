"""GPU parity of the pages' collaboration pruning (Sec. 3.3), the similarity
table (App. A.3, Eq. 8) and the router-logit gradient, through the C ABI.

Expert choices are integer decisions taken on the fp32 logits (and, for
similarity-based pruning, on the fp32 table) by both sides with the same tie
rule, so ids, routed experts and device masks must match bit for bit; gates
carry the fp32 softmax (GATE_RTOL).
"""
import numpy as np
import pytest
import torch

import synth
from layer_cases import assert_close_layer, make_case, reference_output
from oracle import backward as obackward
from oracle import routing as orouting
from oracle import similarity as osim

pytestmark = pytest.mark.gpu

GATE_RTOL = 2e-6
F32_EPS = 2.0 ** -24

BASE = synth.CONFIGS["olmoe_fwd"]
ROUTE_CASES = {
    "olmoe_keep2": BASE.with_(T=3000, limit_devices=2),
    "olmoe_keep3_renorm": BASE.with_(T=2049, limit_devices=3, renorm=True),
    "decode_keep2": synth.CONFIGS["deepseek_decode"].with_(limit_devices=2),
    "ne256_k16": BASE.with_(T=777, n_experts=256, top_k=16, n_vdev=16, limit_devices=2,
                            n_clusters=16, experts_per_cluster=24),
    "ne8_keep1": synth.CONFIGS["tiny_f32"].with_(limit_devices=1),
    "one_token": BASE.with_(T=1, limit_devices=2),
}


@pytest.fixture(scope="module")
def occ():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_top_route_gb300 import build
    build.build()
    import combine_top_route_gb300 as occ
    occ.lib()
    return occ


def _route(occ, cfg, mode, table=None):
    case = make_case(cfg, tensors=False)
    c = cfg.with_(route_mode=mode)
    ds = occ.desc_for(c)
    T, k, Ne = c.T, c.top_k, c.n_experts
    dev = "cuda"
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    gates = torch.empty(T, k, dtype=torch.float32, device=dev)
    vmask = torch.empty(T, dtype=torch.int32, device=dev)
    routed = torch.empty(T, k, dtype=torch.int32, device=dev)
    e2v = torch.as_tensor(case.e2v, dtype=torch.int32, device=dev)
    lg = case.logits.to(dev)
    if mode == "similarity_pruned":
        occ.occult_route_similarity(ds, lg, e2v, table.to(dev), ids, gates, vmask, routed)
    else:
        occ.occult_route(ds, lg, e2v, ids, gates, vmask)
        routed = ids
    torch.cuda.synchronize()
    return case, [t.cpu().numpy() for t in (ids, gates, vmask, routed)]


def _vmask(ids, e2v):
    return np.array([sum(1 << int(d) for d in set(e2v[r].tolist())) for r in ids], dtype=np.int64)


@pytest.mark.parametrize("name", list(ROUTE_CASES))
def test_score_pruned_route(occ, name):
    cfg = ROUTE_CASES[name]
    case, (ids, gates, vmask, _) = _route(occ, cfg, "score_pruned")
    r_ids, r_g, kept = orouting.route_score_pruned(case.logits.numpy(), cfg.top_k, case.e2v,
                                                   cfg.limit_devices, renorm=cfg.renorm)
    np.testing.assert_array_equal(ids, r_ids)
    np.testing.assert_allclose(gates, r_g, rtol=GATE_RTOL)
    np.testing.assert_array_equal(vmask.astype(np.int64) & 0xffffffff, _vmask(r_ids, case.e2v))
    assert max(bin(int(m) & 0xffffffff).count("1") for m in vmask) <= cfg.limit_devices


@pytest.mark.parametrize("name", list(ROUTE_CASES))
def test_similarity_pruned_route(occ, name):
    cfg = ROUTE_CASES[name]
    table = synth.random_similarity_table(cfg)
    case, (ids, gates, vmask, routed) = _route(occ, cfg, "similarity_pruned", table)
    r_ids, r_g, r_routed, _ = orouting.route_similarity_pruned(
        case.logits.numpy(), cfg.top_k, case.e2v, cfg.limit_devices, table.numpy(),
        renorm=cfg.renorm)
    np.testing.assert_array_equal(routed, r_routed)
    np.testing.assert_array_equal(ids, r_ids)
    np.testing.assert_allclose(gates, r_g, rtol=GATE_RTOL)
    np.testing.assert_array_equal(vmask.astype(np.int64) & 0xffffffff, _vmask(r_ids, case.e2v))


@pytest.mark.parametrize("mode", ["score_pruned", "similarity_pruned"])
def test_pruned_layer_output(occ, mode):
    """The whole forward under pruning equals Eq. 1 with the pruned routing."""
    cfg = BASE.with_(T=1536, route_mode=mode, limit_devices=2)
    case = make_case(cfg)
    table = synth.random_similarity_table(cfg) if mode == "similarity_pruned" else None
    moe = occ.OccultMoE(occ.desc_for(cfg), case.weights, torch.as_tensor(case.placement),
                        sim_table=table)
    y = moe.forward(case.logits.cuda(), case.x).cpu().numpy()
    assert occ.device_error() == 0
    ids, gates, _ = case.oracle_route(None if table is None else table.numpy())
    ref = reference_output(case, np.arange(cfg.T), ids, gates.astype(np.float32).astype(np.float64))
    assert_close_layer(y, ref, cfg.dtype)
    n_sfd = int(moe.counts[0].item())
    assert n_sfd <= 2 * cfg.T                       # C_T <= 2 for every token


def test_similarity_table(occ):
    """Eq. 8 accumulated over uneven batches of profiled logits, then finished."""
    cfg = BASE
    ds = occ.desc_for(cfg)
    H = synth.profiling_logits(cfg)
    G = torch.zeros(cfg.n_experts, cfg.n_experts, dtype=torch.float64, device="cuda")
    cuts = [0, 1, 1000, 1000, 7777, H.shape[0]]
    Hd = H.cuda()
    for a, b in zip(cuts[:-1], cuts[1:]):
        occ.occult_similarity_accumulate(ds, Hd[a:b].contiguous(), b - a, G)
    tab = torch.empty(cfg.n_experts, cfg.n_experts, dtype=torch.float32, device="cuda")
    occ.occult_similarity_finish(ds, G, tab)
    torch.cuda.synchronize()
    ref_G = osim.accumulate(np.zeros((cfg.n_experts, cfg.n_experts)), H.numpy())
    np.testing.assert_allclose(G.cpu().numpy(), ref_G, rtol=1e-12, atol=1e-9)
    ref = osim.finish(ref_G)
    got = tab.cpu().numpy().astype(np.float64)
    # fp32 rounding of the fp64 value, plus fp64 summation order
    np.testing.assert_allclose(got, ref, rtol=2 * F32_EPS, atol=1e-12)
    # deterministic: the same batches give the same bits
    G2 = torch.zeros_like(G)
    for a, b in zip(cuts[:-1], cuts[1:]):
        occ.occult_similarity_accumulate(ds, Hd[a:b].contiguous(), b - a, G2)
    assert torch.equal(G, G2)


def _grad_bound(z, ids, dg, renorm):
    """|dz_gpu - dz| bound for fp32 softmax (expf 2 ulp, sums over Ne and k) and the
    few roundings of the formula, per element."""
    p = orouting.softmax(z)
    T, Ne = z.shape
    k = ids.shape[1]
    q = np.take_along_axis(p, ids.astype(int), 1)
    g = q / q.sum(1, keepdims=True) if renorm else q
    A = np.abs(dg * g).sum(1, keepdims=True)
    eps = 4 * (Ne + k + 8) * F32_EPS
    w = np.zeros((T, Ne))
    sel = np.zeros((T, Ne))
    for t in range(T):
        for j in range(k):
            if renorm:
                w[t, ids[t, j]] += g[t, j] * (abs(dg[t, j]) + A[t, 0])
            sel[t, ids[t, j]] += abs(dg[t, j])
    if not renorm:
        w = p * (sel + A)
    return eps * w + 1e-30


@pytest.mark.parametrize("renorm", [False, True])
def test_router_grad(occ, renorm):
    cfg = BASE.with_(T=2500, renorm=renorm)
    case = make_case(cfg, tensors=False)
    z = case.logits.numpy()
    ids, _ = orouting.route_topk(z, cfg.top_k)
    dg = torch.randn(cfg.T, cfg.top_k, generator=torch.Generator().manual_seed(5)).numpy()
    ds = occ.desc_for(cfg)
    out = torch.empty(cfg.T, cfg.n_experts, dtype=torch.float32, device="cuda")
    occ.occult_router_grad(ds, case.logits.cuda(), torch.as_tensor(ids).cuda(),
                           torch.as_tensor(dg).cuda(), out)
    torch.cuda.synchronize()
    ref = obackward.router_grad(z, ids, dg, renorm=renorm)
    err = np.abs(out.cpu().numpy().astype(np.float64) - ref)
    bound = _grad_bound(z.astype(np.float64), ids, dg.astype(np.float64), renorm)
    assert (err <= bound).all(), f"exceeds the bound by up to {float(np.max(err - bound)):.3e}"
    if renorm:
        # unselected experts get exactly nothing
        mask = np.ones_like(ref, dtype=bool)
        np.put_along_axis(mask, ids.astype(int), False, 1)
        assert not out.cpu().numpy()[mask].any()
