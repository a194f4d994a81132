"""Pins of the per-element error bounds that the GPU parity tests use for the
expert FFN's intermediates and gradients (``layer_cases.h_bound``,
``sfd_bound``, ``expert_backward_bounds``), on the CPU.

A CPU emulation of the bf16 GPU arithmetic (``bf16_pipeline``) on the OLMoE
layer's own widths (d = 2048, I = 1024) must
  * stay within every bound, element by element;
  * come within a stated fraction of it (the bound is not vacuous);
and each planted mistake of the kind a kernel bug makes (one EPD row dropped, a
routing weight applied twice, a neighbouring expert's weights) must break the
bounds.  max|diff| / rms of every quantity is printed beside the 2e-2 bar that
the layer output is held to.
"""
import numpy as np
import pytest

import synth
from bf16_pipeline import backward_rows, forward_rows
from layer_cases import (F32_EPS, assert_close_layer, expert_backward_bounds, h_bound,
                         sfd_bound)
from oracle import backward as obackward
from oracle import expert as oexpert
from oracle import routing as orouting

# Smallest worst-case diff / bound the emulation must reach, per quantity: a
# bound far above the error the arithmetic really makes would let a real
# mistake through.  Observed on this layer (and on the full OLMoE training shape,
# k = 8): h 0.38 (0.50), y 0.13 (0.09), dgates 0.064 (0.075), dx 0.072 (0.057),
# dW1 0.57 (0.62), dW2 0.64 (0.68); asserted at about half.  dgates and dx are
# random-walk bounds over sums of 1024 and 2048 rounded terms, built from each
# term's worst rounding and LAMBDA = 10, hence their few per cent.
MIN_RATIO = {"h": 0.2, "y": 0.05, "dg": 0.03, "dx": 0.03, "dW1": 0.25, "dW2": 0.25}

CFG = synth.CONFIGS["olmoe_train"].with_(name="emulation", T=1024, n_experts=8, top_k=2,
                                         n_vdev=4, n_clusters=4, experts_per_cluster=3,
                                         prof_tokens=1024)


@pytest.fixture(scope="module")
def layer():
    cfg = CFG
    x = synth.hidden_states(cfg).float().numpy()
    w = synth.expert_weights(cfg)
    w1, w2 = w["w1"].float().numpy(), w["w2"].float().numpy()
    dy = synth.upstream_grad(cfg).float().numpy()
    ids, gates = orouting.route_topk(synth.measured_logits(cfg).numpy(), cfg.top_k)
    gates = gates.astype(np.float32)             # the GPU's fp32 gates
    ref_y = oexpert.moe_topk(x, ids, gates.astype(np.float64), w1, w2)
    ref_b = obackward.moe_backward(x, ids, gates.astype(np.float64), w1, w2, dy)
    return dict(x=x, w1=w1, w2=w2, dy=dy, ids=ids, gates=gates, ref_y=ref_y, ref_b=ref_b)


def run(layer, mistake=None, mistake_expert=0):
    """The emulated forward and backward of every expert, compared with the oracle
    against the bounds.  Returns {quantity: (ok, worst diff/bound, max|diff|/rms)}."""
    x, w1, w2, dy = layer["x"], layer["w1"], layer["w2"], layer["dy"]
    ids, gates = layer["ids"], layer["gates"]
    T, d = x.shape
    k = ids.shape[1]
    I = w1.shape[1] // 2
    y = np.zeros((T, d), np.float32)
    dx = np.zeros((T, d), np.float32)
    dx_b = np.zeros((T, d))
    dx_abs = np.zeros((T, d))
    h_abs_rows = [[] for _ in range(T)]
    res = {}

    def note(name, got, ref, bound):
        err = np.abs(np.asarray(got, np.float64) - ref)
        ok, worst = bool((err <= bound).all()), float(np.max(err / bound))
        rms = float(np.sqrt(np.mean(ref ** 2)))
        o, w, r = res.get(name, (True, 0.0, 0.0))
        res[name] = (o and ok, max(w, worst), max(r, float(err.max()) / rms))

    for e in range(w1.shape[0]):
        toks, slots = np.nonzero(ids == e)
        if toks.size == 0:
            continue
        a, g = x[toks], gates[toks, slots]
        m = mistake if e == mistake_expert else None
        f = forward_rows(a, w1, w2, e, g, m)
        G = a.astype(np.float64) @ w1[e, :I].T.astype(np.float64)
        U = a.astype(np.float64) @ w1[e, I:].T.astype(np.float64)
        h_ref = g[:, None].astype(np.float64) * oexpert.silu(G) * U
        note("h", f["h"], h_ref, h_bound(a, w1[e, :I], w1[e, I:], g, h_ref, "bf16"))
        y[toks] += f["y_epd"]                   # fp32, slot order within a token
        for i, t in enumerate(toks):
            h_abs_rows[t].append((e, np.abs(h_ref[i])))
        b = expert_backward_bounds(a, dy[toks], w1[e], w2[e], g)
        r = backward_rows(a, dy[toks], w1, w2, e, g, f, m)
        note("dg", r["dg"], layer["ref_b"]["dgates"][toks, slots], b["dg_b"])
        note("dW1", r["dW1"], layer["ref_b"]["dw1"][e], b["dW1_b"] + 1e-30)
        note("dW2", r["dW2"], layer["ref_b"]["dw2"][e], b["dW2_b"] + 1e-30)
        dx[toks] += r["dx_rows"]
        dx_b[toks] += b["dx_rows_b"]
        dx_abs[toks] += np.abs(b["dx_rows"]) + b["dx_rows_b"]
    # a token's k rows summed in fp32: the SFD-row bound over all of its rows
    y_b = np.stack([sfd_bound(w2, h_abs_rows[t], "bf16") for t in range(T)])
    note("y", y, layer["ref_y"], y_b + 1e-30)
    note("dx", dx, layer["ref_b"]["dx"], dx_b + 2 * k * F32_EPS * dx_abs + 1e-30)
    return res, y


def test_bounds_hold_and_are_not_vacuous(layer):
    res, y = run(layer)
    for name, (ok, worst, rel) in sorted(res.items()):
        print(f"{name}: max|diff|/rms {rel:.4f} (layer-output bar 0.02), worst diff/bound {worst:.3f}")
    for name, (ok, worst, _) in res.items():
        assert ok, f"{name}: the emulated bf16 arithmetic exceeds its bound"
        assert worst >= MIN_RATIO[name], f"{name}: bound vacuous, worst diff/bound {worst:.3f}"
    # the layer output meets the 2e-2 * rms bar as well
    assert_close_layer(y, layer["ref_y"], "bf16")


@pytest.mark.parametrize("mistake", ["drop_row", "gate_twice", "neighbour"])
def test_planted_mistakes_break_the_bounds(layer, mistake):
    counts = np.bincount(layer["ids"].ravel(), minlength=CFG.n_experts)
    e = int(np.argmax(counts))      # the busiest expert: the mistake is diluted most
    res, _ = run(layer, mistake, e)
    for name in ("h", "y", "dx"):
        assert not res[name][0], f"{mistake}: {name} still within its bound"
    if mistake != "drop_row":
        # every row of the expert is wrong: its weight gradients too
        assert not res["dW1"][0] and not res["dW2"][0]
    if mistake == "neighbour":
        # (dgates = <dh', h> does not involve the routing weight itself)
        assert not res["dg"][0]
