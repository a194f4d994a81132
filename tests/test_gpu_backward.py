"""GPU parity of the layer's backward against the fp64 oracle, through the C ABI.

The weight gradients contract bf16 operands that the forward rounded (h' and the
saved G, U) and that the backward rounds (dG, dU); no bf16 tensor-core backward
meets a 2e-2 * rms bar on them element by element (a CPU emulation gives
0.11-0.15 * rms), so every output is checked against per-element bounds derived
from that arithmetic (layer_cases.expert_backward_bounds), and max|diff| / rms
is reported beside.  The 1024-token slice of the training workload and a
ragged small layer are checked completely; the full 32768-token step on
sampled tokens and experts.
"""
import numpy as np
import pytest
import torch

import synth
from layer_cases import F32_EPS, expert_backward_bounds, make_case
from oracle import backward as obackward

pytestmark = pytest.mark.gpu

TRAIN = synth.CONFIGS["olmoe_train"]
CASES = {
    "train_slice_1024": TRAIN.with_(name="train_slice_1024", T=1024),
    "ragged_i192": TRAIN.with_(name="ragged_i192", T=333, d=512, inter=192, n_vdev=8),
    # >= 256 rows an expert: the dgrads run on CTA pairs
    "pair_ragged": TRAIN.with_(name="pair_ragged", T=2600, d=512, inter=192, n_vdev=8),
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


def train_step(occ, case, dy, merge=None):
    moe = occ.OccultMoE(occ.desc_for(case.cfg), case.weights, torch.as_tensor(case.placement),
                        train=True, merge=merge)
    moe.forward(case.logits.cuda(), case.x)
    out = moe.backward(dy)
    torch.cuda.synchronize()
    assert occ.device_error() == 0
    return moe, [t.cpu().numpy() for t in out]


def check(name, got, ref, bound):
    err = np.abs(got.astype(np.float64) - ref)
    rms = float(np.sqrt(np.mean(ref ** 2))) or 1.0
    worst = float(np.max(err / bound)) if err.size else 0.0
    print(f"{name}: max|diff|/rms {float(err.max()) / rms:.4f}, worst diff/bound {worst:.3f}")
    assert (err <= bound).all(), f"{name}: exceeds its bound by up to {float(np.max(err - bound)):.3e}"


def bounds_for_rows(case, ids, gates, dy_h, rows_of_expert):
    """Per-(token, slot) bounds from the expert-wise arithmetic bounds."""
    x = case.host("x")
    w1, w2 = case.host("w1"), case.host("w2")
    out = {}
    for e, (toks, slots) in rows_of_expert.items():
        out[e] = (toks, slots, expert_backward_bounds(x[toks], dy_h[toks], w1[e], w2[e],
                                                      gates[toks, slots]))
    return out


@pytest.mark.parametrize("name", list(CASES))
def test_backward_full_check(occ, name):
    cfg = CASES[name]
    case = make_case(cfg)
    dy = synth.upstream_grad(cfg, device="cuda")
    moe, (dx, dw1, dw2, dgates) = train_step(occ, case, dy)
    ids, gates, _ = case.oracle_route()
    gates = gates.astype(np.float32).astype(np.float64)  # the GPU's fp32 gates
    dy_h = dy.float().cpu().numpy()
    ref = obackward.moe_backward(case.host("x"), ids, gates, case.host("w1"), case.host("w2"), dy_h)
    rows = {int(e): np.nonzero(ids == e) for e in np.unique(ids)}
    B = bounds_for_rows(case, ids, gates, dy_h, rows)
    T, k, d = cfg.T, cfg.top_k, cfg.d
    dx_b = np.zeros((T, d))
    dx_abs = np.zeros((T, d))
    dg_b = np.zeros((T, k))
    for e, (toks, slots, b) in B.items():
        np.add.at(dx_b, toks, b["dx_rows_b"])
        np.add.at(dx_abs, toks, np.abs(b["dx_rows"]) + b["dx_rows_b"])
        dg_b[toks, slots] = b["dg_b"]
    dx_b += 2 * k * F32_EPS * dx_abs          # the fp32 two-stage merge
    check("dx", dx, ref["dx"], dx_b + 1e-30)
    check("dgates", dgates, ref["dgates"], dg_b)
    # router logits: the oracle's d-logits of the oracle's dgates; the GPU's carry
    # the dgates error through p_e (sel_e - A), plus their own fp32 rounding
    z = case.logits.numpy().astype(np.float64)
    dz_ref = obackward.router_grad(z, ids, ref["dgates"])
    p = np.exp(z - z.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    g = np.take_along_axis(p, ids.astype(int), 1)
    sel_b = np.zeros_like(z)
    sel_a = np.zeros_like(z)
    for j in range(k):
        np.add.at(sel_b, (np.arange(T), ids[:, j]), dg_b[:, j])
        np.add.at(sel_a, (np.arange(T), ids[:, j]), np.abs(ref["dgates"][:, j]) + dg_b[:, j])
    A_b = (dg_b * g).sum(1, keepdims=True)
    A_a = ((np.abs(ref["dgates"]) + dg_b) * g).sum(1, keepdims=True)
    dz_b = p * (sel_b + A_b) + 4 * (cfg.n_experts + k + 8) * F32_EPS * p * (sel_a + A_a) + 1e-30
    check("dlogits", moe.dlogits.cpu().numpy(), dz_ref, dz_b)
    w1_b = np.zeros_like(ref["dw1"])
    w2_b = np.zeros_like(ref["dw2"])
    for e, (_, _, b) in B.items():
        w1_b[e], w2_b[e] = b["dW1_b"], b["dW2_b"]
    unused = [e for e in range(cfg.n_experts) if e not in B]
    assert all(not dw1[e].any() and not dw2[e].any() for e in unused), "an unused expert's gradient is not zero"
    used = sorted(B)
    check("dW1", dw1[used], ref["dw1"][used], w1_b[used] + 1e-30)
    check("dW2", dw2[used], ref["dw2"][used], w2_b[used] + 1e-30)


def test_backward_full_size_sampled(occ):
    """The whole 32768-token training step; sampled tokens and experts checked."""
    cfg = TRAIN
    case = make_case(cfg)
    dy = synth.upstream_grad(cfg, device="cuda")
    moe, (dx, dw1, dw2, dgates) = train_step(occ, case, dy)
    ids, gates, _ = case.oracle_route()
    gates = gates.astype(np.float32).astype(np.float64)
    dy_h = dy.float().cpu().numpy()
    x, w1, w2 = case.host("x"), case.host("w1"), case.host("w2")
    rng = np.random.default_rng(3)
    toks = np.unique(np.concatenate([np.arange(8), rng.choice(cfg.T, 56, replace=False),
                                     [cfg.T - 1]]))
    # tokens: dx and dgates from the oracle on those rows (rows are independent)
    sub = obackward.moe_backward(x[toks], ids[toks], gates[toks], w1, w2, dy_h[toks])
    k, d = cfg.top_k, cfg.d
    dx_b = np.zeros((toks.size, d))
    dx_abs = np.zeros((toks.size, d))
    dg_b = np.zeros((toks.size, k))
    for e in np.unique(ids[toks]):
        r, sl = np.nonzero(ids[toks] == e)
        b = expert_backward_bounds(x[toks][r], dy_h[toks][r], w1[e], w2[e], gates[toks][r, sl])
        np.add.at(dx_b, r, b["dx_rows_b"])
        np.add.at(dx_abs, r, np.abs(b["dx_rows"]) + b["dx_rows_b"])
        dg_b[r, sl] = b["dg_b"]
    dx_b += 2 * k * F32_EPS * dx_abs
    check("dx[sampled]", dx[toks], sub["dx"], dx_b + 1e-30)
    check("dgates[sampled]", dgates[toks], sub["dgates"], dg_b)
    # experts: all rows of a few experts
    counts = np.bincount(ids.ravel(), minlength=cfg.n_experts)
    for e in [int(np.argmax(counts)), int(np.argmin(counts)), int(case.placement[-1, -1])]:
        te, se = np.nonzero(ids == e)
        ref = obackward.moe_backward(x[te], ids[te], gates[te], w1, w2, dy_h[te], experts=[e])
        b = expert_backward_bounds(x[te], dy_h[te], w1[e], w2[e], gates[te, se])
        check(f"dW1[{e}]", dw1[e], ref["dw1"][e], b["dW1_b"] + 1e-30)
        check(f"dW2[{e}]", dw2[e], ref["dw2"][e], b["dW2_b"] + 1e-30)


@pytest.mark.parametrize("name", list(CASES))
def test_atomic_and_ordered_merges_agree(occ, name):
    """The merge only changes the order of dx's fp32 additions: the weight and gate
    gradients are bit for bit the same, dx within 2 k 2^-24 sum|rows| (the sum of
    |rows| taken from the ordered run's fp32 EPD rows)."""
    cfg = CASES[name]
    case = make_case(cfg)
    dy = synth.upstream_grad(cfg, device="cuda")
    moe_o, out_o = train_step(occ, case, dy, merge="ordered")
    dx_abs = np.zeros((cfg.T, cfg.d))
    tok = moe_o.sfd_tok.cpu().numpy()[moe_o.epd_src.cpu().numpy()]
    np.add.at(dx_abs, tok, np.abs(moe_o.dx_epd.cpu().numpy().astype(np.float64)))
    moe_a, out_a = train_step(occ, case, dy, merge="atomic")
    assert moe_a.merge == "atomic" and moe_a.dx_epd is None
    for a, b, nm in zip(out_a[1:], out_o[1:], ("dw1", "dw2", "dgates")):
        assert (a == b).all(), nm
    assert (moe_a.dlogits.cpu().numpy() == moe_o.dlogits.cpu().numpy()).all()
    err = np.abs(out_a[0].astype(np.float64) - out_o[0])
    assert (err <= 2 * cfg.top_k * F32_EPS * dx_abs + 1e-30).all()
