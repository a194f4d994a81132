"""Pins of the oracle layer output (Eq. 1) against closed forms and an
independent torch-CPU formulation."""
import numpy as np
import pytest
import torch

from oracle import expert, routing


def test_scalar_swiglu_closed_form(golden):
    g = golden("closed_forms.json")["swiglu_scalar"]
    w1 = np.array([[[g["w_g"]], [g["w_u"]]]])
    w2 = np.array([[[g["w_d"]]]])
    y = expert.moe_topk(np.array([[g["x"]]]), np.array([[0]]), np.array([[1.0]]), w1, w2)
    assert abs(y[0, 0] - g["y"]) < 1e-14


def test_zero_input_gives_zero():
    rng = np.random.default_rng(0)
    w1 = rng.standard_normal((4, 6, 5))
    w2 = rng.standard_normal((4, 5, 3))
    y = expert.moe_topk(np.zeros((3, 5)), np.array([[0, 1]] * 3), np.ones((3, 2)), w1, w2)
    assert (y == 0).all()


def test_linear_in_gates():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 5))
    w1 = rng.standard_normal((4, 6, 5))
    w2 = rng.standard_normal((4, 5, 3))
    ids = np.array([[0, 2]] * 7)
    g = rng.random((7, 2))
    y = expert.moe_topk(x, ids, g, w1, w2)
    y1 = expert.moe_topk(x, ids, g * np.array([1.0, 0.0]), w1, w2)
    y2 = expert.moe_topk(x, ids, g * np.array([0.0, 1.0]), w1, w2)
    np.testing.assert_allclose(y, y1 + y2, rtol=1e-13, atol=1e-14)


def test_token_subset_matches_full():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((20, 6))
    logits = rng.standard_normal((20, 5)).astype(np.float32)
    ids, g = routing.route_topk(logits, 2)
    w1 = rng.standard_normal((5, 8, 6))
    w2 = rng.standard_normal((5, 6, 4))
    y = expert.moe_topk(x, ids, g, w1, w2)
    sub = [17, 3, 9]
    np.testing.assert_allclose(expert.moe_topk(x, ids, g, w1, w2, sub), y[sub], rtol=1e-14)


def test_matches_torch_autograd_free_formulation():
    """Independent torch-CPU einsum formulation of the same layer (fp64)."""
    rng = np.random.default_rng(3)
    T, d, Ne, I, k = 33, 16, 6, 12, 3
    x = rng.standard_normal((T, d))
    logits = rng.standard_normal((T, Ne)).astype(np.float32)
    ids, g = routing.route_topk(logits, k, renorm=True)
    w1 = rng.standard_normal((Ne, 2 * I, d)) * 0.2
    w2 = rng.standard_normal((Ne, d, I)) * 0.2
    y = expert.moe_topk(x, ids, g, w1, w2)
    tx, tw1, tw2 = map(torch.from_numpy, (x, w1, w2))
    W = tw1[torch.from_numpy(ids.astype(np.int64))]          # [T, k, 2I, d]
    hg = torch.einsum("tkid,td->tki", W[:, :, :I], tx)
    hu = torch.einsum("tkid,td->tki", W[:, :, I:], tx)
    h = torch.nn.functional.silu(hg) * hu
    out = torch.einsum("tkdi,tki->tkd", tw2[torch.from_numpy(ids.astype(np.int64))], h)
    yt = (out * torch.from_numpy(g)[:, :, None]).sum(1).numpy()
    np.testing.assert_allclose(y, yt, rtol=1e-12, atol=1e-13)


def test_shared_gate_zero_vector_is_one_half():
    x = np.random.default_rng(4).standard_normal((5, 3))
    np.testing.assert_array_equal(expert.shared_gate(x, np.zeros(3)), np.full(5, 0.5))


def test_stacked_shared_experts_equal_their_sum():
    """Two shared experts equal one expert over their concatenated hidden units."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((9, 4))
    a1, b1 = rng.standard_normal((6, 4)), rng.standard_normal((6, 4))   # [2I, d] each, I = 3
    a2, b2 = rng.standard_normal((4, 3)), rng.standard_normal((4, 3))   # [d, I]
    ws1 = np.concatenate([a1[:3], b1[:3], a1[3:], b1[3:]])
    ws2 = np.concatenate([a2, b2], axis=1)
    y = expert.shared_experts(x, ws1, ws2)
    ref = expert.swiglu_expert(x, a1, a2) + expert.swiglu_expert(x, b1, b2)
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-14)


def test_shared_gate_closed_form(golden):
    """sigmoid of +ln 3 is 3/4 and of -ln 3 is 1/4: a flipped sign swaps them."""
    g = golden("closed_forms.json")["shared_gate"]
    x = np.array(g["x"])
    np.testing.assert_allclose(expert.shared_gate(x, np.array(g["w_sg_pos"])), g["s_pos"],
                               rtol=1e-15)
    np.testing.assert_allclose(expert.shared_gate(x, np.array(g["w_sg_neg"])), g["s_neg"],
                               rtol=1e-14)


def test_shared_expert_scalar_closed_form(golden):
    g = golden("closed_forms.json")["shared_expert_scalar"]
    ws1 = np.array([[g["w_g"]], [g["w_u"]]])
    ws2 = np.array([[g["w_d"]]])
    y = expert.shared_experts(np.array([[g["x"]]]), ws1, ws2, np.array([g["w_sg"]]))
    assert abs(y[0, 0] - g["y"]) < 1e-14
    # the layer output adds it to the routed experts' Eq. 1 sum
    w = {"w1": ws1[None], "w2": ws2[None], "ws1": ws1, "ws2": ws2, "w_sg": np.array([g["w_sg"]])}
    routed = expert.moe_topk(np.array([[g["x"]]]), np.array([[0]]), np.array([[1.0]]),
                             w["w1"], w["w2"])
    out = expert.layer_output(np.array([[g["x"]]]), np.array([[0]]), np.array([[1.0]]), w)
    assert abs(out[0, 0] - (routed[0, 0] + g["y"])) < 1e-14


@pytest.mark.parametrize("gated", [True, False])
def test_shared_experts_match_torch_formulation(gated):
    """Independent torch-CPU formulation of two stacked shared experts, with and
    without the sigmoid gate (fp64): each expert computed on its own rows of the
    stacked weights and summed."""
    rng = np.random.default_rng(6)
    T, d, I = 11, 8, 5
    x = rng.standard_normal((T, d))
    e1 = rng.standard_normal((2 * I, d)) * 0.3, rng.standard_normal((d, I)) * 0.3
    e2 = rng.standard_normal((2 * I, d)) * 0.3, rng.standard_normal((d, I)) * 0.3
    # stacked along the intermediate axis: gate rows of both, then up rows of both
    ws1 = np.concatenate([e1[0][:I], e2[0][:I], e1[0][I:], e2[0][I:]])
    ws2 = np.concatenate([e1[1], e2[1]], axis=1)
    w_sg = rng.standard_normal(d) if gated else None
    y = expert.shared_experts(x, ws1, ws2, w_sg)
    tx = torch.from_numpy(x)
    out = torch.zeros(T, d, dtype=torch.float64)
    for a, b in (e1, e2):
        ta, tb = torch.from_numpy(a), torch.from_numpy(b)
        out += torch.nn.functional.linear(
            torch.nn.functional.silu(torch.nn.functional.linear(tx, ta[:I]))
            * torch.nn.functional.linear(tx, ta[I:]), tb)
    if gated:
        out = torch.sigmoid(tx @ torch.from_numpy(w_sg))[:, None] * out
    np.testing.assert_allclose(y, out.numpy(), rtol=1e-12, atol=1e-13)
