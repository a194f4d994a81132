"""GPU parity of the layer's backward against the fp64 oracle, through the C ABI.

The weight gradients contract bf16 operands that the forward rounded (h' and the
saved G, U) and that the backward rounds (dG, dU); no bf16 tensor-core backward
meets a 2e-2 * rms bar on them element by element (a CPU emulation gives
0.11-0.15 * rms), so every output is checked against per-element bounds derived
from that arithmetic (layer_cases.expert_backward_bounds), and max|diff| / rms
is reported beside.  Every case is checked completely: the 1024-token slice of
the training workload, ragged small layers and the full 32768-token step.
"""
import numpy as np
import pytest
import torch

import synth
from layer_cases import F32_EPS, expert_backward_bounds, make_case, scatter_add_rows
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


class Checker:
    """Element-wise comparison against per-element bounds, accumulated over pieces
    of one gradient (the weight gradients are checked expert by expert); prints
    max|diff| / rms(ref) beside the 2e-2 bar of the layer output and the worst
    diff / bound."""

    def __init__(self, name):
        self.name, self.err, self.sq, self.n, self.worst = name, 0.0, 0.0, 0, 0.0

    def add(self, got, ref, bound, where=""):
        err = np.abs(got.astype(np.float64) - ref)
        if err.size:
            self.err = max(self.err, float(err.max()))
            self.sq += float(np.sum(ref ** 2))
            self.n += ref.size
            self.worst = max(self.worst, float(np.max(err / bound)))
        assert (err <= bound).all(), (
            f"{self.name}{where}: exceeds its bound by up to {float(np.max(err - bound)):.3e}")

    def report(self):
        rms = np.sqrt(self.sq / max(self.n, 1)) or 1.0
        print(f"{self.name}: max|diff|/rms {self.err / rms:.4f} (layer-output bar 0.02), "
              f"worst diff/bound {self.worst:.3f}")


def check(name, got, ref, bound):
    c = Checker(name)
    c.add(got, ref, bound)
    c.report()


def full_backward_check(case, dy_h, dx, dw1, dw2, dgates, dlogits):
    """Every element of dx, dgates, d-logits, dW1 and dW2 against the fp64 oracle
    (Eq. 1's derivative over the whole batch), each within the bound derived from
    the arithmetic of its rows.  Experts are visited one at a time, so that the
    bounds' intermediates of one expert are held at once."""
    cfg = case.cfg
    ids, gates, _ = case.oracle_route()
    gates = gates.astype(np.float32).astype(np.float64)  # the GPU's fp32 gates
    x, w1, w2 = case.host("x"), case.host("w1"), case.host("w2")
    ref = obackward.moe_backward(x, ids, gates, w1, w2, dy_h)
    T, k, d = cfg.T, cfg.top_k, cfg.d
    dx_b = np.zeros((T, d))
    dx_abs = np.zeros((T, d))
    dg_b = np.zeros((T, k))
    c_w1, c_w2 = Checker("dW1"), Checker("dW2")
    used = [int(e) for e in np.unique(ids)]
    for e in used:
        toks, slots = np.nonzero(ids == e)     # a token holds an expert at most once
        b = expert_backward_bounds(x[toks], dy_h[toks], w1[e], w2[e], gates[toks, slots])
        dx_b[toks] += b["dx_rows_b"]
        dx_abs[toks] += np.abs(b["dx_rows"]) + b["dx_rows_b"]
        dg_b[toks, slots] = b["dg_b"]
        c_w1.add(dw1[e], ref["dw1"][e], b["dW1_b"] + 1e-30, f"[{e}]")
        c_w2.add(dw2[e], ref["dw2"][e], b["dW2_b"] + 1e-30, f"[{e}]")
    c_w1.report()
    c_w2.report()
    unused = [e for e in range(cfg.n_experts) if e not in set(used)]
    assert all(not dw1[e].any() and not dw2[e].any() for e in unused), (
        "an unused expert's gradient is not zero")
    dx_b += 2 * k * F32_EPS * dx_abs          # the fp32 merge of a token's rows
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
    rows = np.arange(T)
    for j in range(k):
        sel_b[rows, ids[:, j]] += dg_b[:, j]      # a token's ids are distinct
        sel_a[rows, ids[:, j]] += np.abs(ref["dgates"][:, j]) + dg_b[:, j]
    A_b = (dg_b * g).sum(1, keepdims=True)
    A_a = ((np.abs(ref["dgates"]) + dg_b) * g).sum(1, keepdims=True)
    dz_b = p * (sel_b + A_b) + 4 * (cfg.n_experts + k + 8) * F32_EPS * p * (sel_a + A_a) + 1e-30
    check("dlogits", dlogits, dz_ref, dz_b)


def run_and_check(occ, cfg):
    case = make_case(cfg)
    dy = synth.upstream_grad(cfg, device="cuda")
    moe, (dx, dw1, dw2, dgates) = train_step(occ, case, dy)
    dlogits = moe.dlogits.cpu().numpy()
    del moe
    full_backward_check(case, dy.float().cpu().numpy(), dx, dw1, dw2, dgates, dlogits)


@pytest.mark.parametrize("name", list(CASES))
def test_backward_full_check(occ, name):
    run_and_check(occ, CASES[name])


def test_backward_full_size(occ):
    """The whole 32768-token training step, every gradient element checked."""
    run_and_check(occ, TRAIN)


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
    scatter_add_rows(dx_abs, tok, np.abs(moe_o.dx_epd.cpu().numpy().astype(np.float64)))
    moe_a, out_a = train_step(occ, case, dy, merge="atomic")
    assert moe_a.merge == "atomic" and moe_a.dx_epd is None
    for a, b, nm in zip(out_a[1:], out_o[1:], ("dw1", "dw2", "dgates")):
        assert (a == b).all(), nm
    assert (moe_a.dlogits.cpu().numpy() == moe_o.dlogits.cpu().numpy()).all()
    err = np.abs(out_a[0].astype(np.float64) - out_o[0])
    assert (err <= 2 * cfg.top_k * F32_EPS * dx_abs + 1e-30).all()


def padded_rows(occ, moe):
    """Row of the padded EPD copy that every EPD row goes to, and the copy's
    zero padding rows (up to a whole number of EPD_PAD rows a slot)."""
    off = moe.exp_off.cpu().numpy().astype(np.int64)
    n = np.diff(off)
    slot = np.repeat(np.arange(n.size), n)
    prow = np.arange(off[-1]) + occ.EPD_PAD * slot
    pad = [np.arange(off[s] + occ.EPD_PAD * s + n[s],
                     off[s] + occ.EPD_PAD * s + -(-n[s] // occ.EPD_PAD) * occ.EPD_PAD)
           for s in range(n.size)]
    return torch.as_tensor(prow, device="cuda"), torch.as_tensor(np.concatenate(pad),
                                                                 device="cuda")


@pytest.mark.parametrize("name", list(CASES))
def test_padded_epd_copies(occ, name):
    """The padded EPD layouts: EPD row r of slot s at row r + EPD_PAD s, zeros
    after each slot's rows up to a whole number of EPD_PAD rows (what the weight
    gradients read past a slot's end).  x_epd, written by the training
    up-projection from the rows it gathers, holds x_sfd[epd_src[r]] bit for bit;
    dy_epd, written by occult_dispatch_epd straight from dy, holds dy[token of r]
    (the token of SFD row epd_src[r], as occult_dispatch numbered them)."""
    cfg = CASES[name]
    case = make_case(cfg)
    dy = synth.upstream_grad(cfg, device="cuda")
    moe, _ = train_step(occ, case, dy)
    prow, pad = padded_rows(occ, moe)
    src = moe.epd_src.long()
    assert torch.equal(moe.x_epd[prow], moe.x_sfd[src])
    assert torch.equal(moe.dy_epd[prow], dy[moe.sfd_tok.long()[src]])
    assert pad.numel() > 0
    assert not moe.x_epd[pad].any() and not moe.dy_epd[pad].any()


@pytest.mark.parametrize("name,T", [("deepseek_decode_limited", 512), ("olmoe_fwd_score_pruned", 1024),
                                    ("olmoe_fwd", 3)])
def test_dispatch_epd_under_other_routings(occ, name, T):
    """occult_dispatch_epd follows the EPD numbering the BRIM build gives under
    device-limited and score-pruned routing, and on a 3-token batch where most
    experts get no row (no padding then): every EPD row holds dy[token of the
    row] bit for bit, every padding row zero; T = 0 is accepted and writes
    nothing."""
    cfg = synth.CONFIGS[name].with_(T=T)
    case = make_case(cfg)
    ds = occ.desc_for(cfg)
    moe = occ.OccultMoE(ds, case.weights, torch.as_tensor(case.placement))
    moe.forward(case.logits.cuda(), case.x)
    dy = synth.upstream_grad(cfg, device="cuda")
    dy_epd = torch.full((occ.epd_copy_rows(ds), cfg.d), float("nan"), dtype=torch.bfloat16,
                        device="cuda")
    occ.occult_dispatch_epd(ds, dy, moe.ids, moe.placement, moe.brim0, moe.seg_off, moe.brim1,
                            moe.exp_off, dy_epd)
    torch.cuda.synchronize()
    assert occ.device_error() == 0
    prow, pad = padded_rows(occ, moe)
    assert torch.equal(dy_epd[prow], dy[moe.sfd_tok.long()[moe.epd_src.long()]])
    assert not dy_epd[pad].any()
    before = dy_epd.clone()
    empty = occ.desc_for(cfg.with_(T=0))
    occ.occult_dispatch_epd(empty, dy[:0], moe.ids[:0], moe.placement, moe.brim0, moe.seg_off,
                            moe.brim1, moe.exp_off, dy_epd)
    torch.cuda.synchronize()
    assert torch.equal(dy_epd.view(torch.int16), before.view(torch.int16))


@pytest.mark.parametrize("name", ["train_slice_1024", "pair_ragged"])
def test_split_backward_equals_fused(occ, name):
    """The four backward GEMMs called one by one (occult_expert_dgrad_down,
    _dgrad_up, _wgrad_down, _wgrad_up) give the fused call's results: the weight
    and gate gradients bit for bit, whether the GEMMs gather dy and x rows from
    the SFD buffers (dy dispatched with occult_dispatch here) or read the padded
    EPD layouts as tiles; dx (fp32 atomic adds in no fixed order) within
    2 k 2^-24 sum|rows|; so does the ordered form (EPD rows + combine)."""
    cfg = CASES[name]
    case = make_case(cfg)
    dy = synth.upstream_grad(cfg, device="cuda")
    moe, (dx, dw1, dw2, dgates) = train_step(occ, case, dy)   # the fused call
    ds = moe.desc
    dg_epd = moe.dg_epd.clone()
    dgu_fused = moe.dgu_epd.clone()
    # dy's SFD rows, as the sharded path and the gathering GEMMs take them
    dy_sfd = torch.empty_like(moe.x_sfd)
    occ.occult_dispatch(ds, dy, moe.brim0, moe.vmask, dy_sfd)
    # dh' from dy's padded EPD rows (the fused call's input), once more
    dgu_t = torch.empty_like(moe.dgu_epd)
    dg_t = torch.empty_like(moe.dg_epd)
    occ.occult_expert_dgrad_down(ds, None, moe.epd_src, moe.epd_gate, moe.exp_off, moe.placement,
                                 moe.w["w2"], moe.gu_epd, dgu_t, dg_t, moe.bwd_ws,
                                 dy_epd=moe.dy_epd)
    dgu = torch.empty_like(moe.dgu_epd)
    dg2 = torch.empty_like(moe.dg_epd)
    dy_epd = torch.full_like(moe.dy_epd, float("nan"))
    dx2 = torch.full_like(moe.dx, float("nan"))
    dw1_2 = torch.full_like(moe.dw1, float("nan"))
    dw2_2 = torch.full_like(moe.dw2, float("nan"))
    occ.occult_expert_dgrad_down(ds, dy_sfd, moe.epd_src, moe.epd_gate, moe.exp_off,
                                 moe.placement, moe.w["w2"], moe.gu_epd, dgu, dg2, moe.bwd_ws,
                                 dy_epd=dy_epd)
    occ.occult_expert_dgrad_up(ds, dgu, moe.epd_src, moe.exp_off, moe.placement, moe.w["w1"],
                               dx2, sfd_tok=moe.sfd_tok, zero_dx=True)
    occ.occult_expert_wgrad_down(ds, dy_sfd, moe.epd_src, moe.exp_off, moe.placement,
                                 moe.h_epd, dw2_2)
    occ.occult_expert_wgrad_up(ds, moe.x_sfd, moe.epd_src, moe.exp_off, moe.placement, dgu,
                               dw1_2)
    # the same from the padded EPD copies (the SFD buffers not passed)
    dw1_3 = torch.full_like(moe.dw1, float("nan"))
    dw2_3 = torch.full_like(moe.dw2, float("nan"))
    occ.occult_expert_wgrad_down(ds, None, None, moe.exp_off, moe.placement, moe.h_epd, dw2_3,
                                 dy_epd=dy_epd)
    occ.occult_expert_wgrad_up(ds, None, None, moe.exp_off, moe.placement, dgu, dw1_3,
                               x_epd=moe.x_epd)
    # the ordered form: fp32 EPD rows, merged by the combine
    dx_epd = torch.empty(cfg.T * cfg.top_k, cfg.d, dtype=torch.float32, device="cuda")
    occ.occult_expert_dgrad_up(ds, dgu, moe.epd_src, moe.exp_off, moe.placement, moe.w["w1"],
                               dx_epd)
    dx3 = torch.empty_like(moe.dx)
    occ.occult_combine(ds, dx_epd, moe.brim0, moe.seg_off, moe.brim1, moe.exp_off, dx3)
    torch.cuda.synchronize()
    assert occ.device_error() == 0
    assert torch.equal(dgu, dgu_fused) and torch.equal(dg2, dg_epd)
    assert torch.equal(dgu_t, dgu_fused) and torch.equal(dg_t, dg_epd)
    assert (dw1_2.cpu().numpy() == dw1).all() and (dw2_2.cpu().numpy() == dw2).all()
    assert (dw1_3.cpu().numpy() == dw1).all() and (dw2_3.cpu().numpy() == dw2).all()
    prow, _ = padded_rows(occ, moe)
    assert torch.equal(dy_epd[prow], moe.dy_epd[prow])
    dx_abs = np.zeros((cfg.T, cfg.d))
    tok = moe.sfd_tok.cpu().numpy()[moe.epd_src.cpu().numpy()]
    scatter_add_rows(dx_abs, tok, np.abs(dx_epd.cpu().numpy().astype(np.float64)))
    bound = 2 * cfg.top_k * F32_EPS * dx_abs + 1e-30
    for got in (dx2, dx3):
        err = np.abs(got.cpu().numpy().astype(np.float64) - dx)
        assert (err <= bound).all()
