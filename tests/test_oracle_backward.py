"""Pins of the oracle backward against central finite differences of the oracle's
own forward (Eq. 1) and an independent torch-CPU autograd formulation."""
import numpy as np
import pytest
import torch

from oracle import backward, expert, routing


def _case(seed, T=6, d=5, Ne=4, I=3, k=2):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    logits = rng.standard_normal((T, Ne)).astype(np.float32)
    ids, gates = routing.route_topk(logits, k, renorm=True)
    w1 = rng.standard_normal((Ne, 2 * I, d)) * 0.5
    w2 = rng.standard_normal((Ne, d, I)) * 0.5
    dy = rng.standard_normal((T, d))
    return x, ids, gates, w1, w2, dy


def _loss(x, ids, gates, w1, w2, dy):
    return float(np.sum(dy * expert.moe_topk(x, ids, gates, w1, w2)))


@pytest.mark.parametrize("seed", [0, 1])
def test_matches_central_differences(seed):
    x, ids, gates, w1, w2, dy = _case(seed)
    g = backward.moe_backward(x, ids, gates, w1, w2, dy)
    eps = 1e-6

    def fd(arr, f):
        out = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            old = arr[i]
            arr[i] = old + eps
            lp = f()
            arr[i] = old - eps
            lm = f()
            arr[i] = old
            out[i] = (lp - lm) / (2 * eps)
        return out

    f = lambda: _loss(x, ids, gates, w1, w2, dy)  # noqa: E731
    np.testing.assert_allclose(g["dx"], fd(x, f), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(g["dw1"], fd(w1, f), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(g["dw2"], fd(w2, f), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(g["dgates"], fd(gates, f), rtol=1e-6, atol=1e-8)


def test_matches_torch_autograd():
    x, ids, gates, w1, w2, dy = _case(3, T=20, d=8, Ne=6, I=5, k=3)
    g = backward.moe_backward(x, ids, gates, w1, w2, dy)
    tx, tw1, tw2, tg = (torch.tensor(a, requires_grad=True) for a in (x, w1, w2, gates))
    I = w1.shape[1] // 2
    idx = torch.as_tensor(ids.astype(np.int64))
    W = tw1[idx]                                   # [T, k, 2I, d]
    hg = torch.einsum("tkid,td->tki", W[:, :, :I], tx)
    hu = torch.einsum("tkid,td->tki", W[:, :, I:], tx)
    h = torch.nn.functional.silu(hg) * hu
    out = torch.einsum("tkdi,tki->tkd", tw2[idx], h)
    y = (out * tg[:, :, None]).sum(1)
    (y * torch.as_tensor(dy)).sum().backward()
    np.testing.assert_allclose(g["dx"], tx.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(g["dw1"], tw1.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(g["dw2"], tw2.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(g["dgates"], tg.grad.numpy(), rtol=1e-11, atol=1e-12)


def test_gate_gradient_is_expert_output_dot_dy():
    """y is linear in each gate: dL/dg_tj = <dy_t, E_e(x_t)>."""
    x, ids, gates, w1, w2, dy = _case(4)
    g = backward.moe_backward(x, ids, gates, w1, w2, dy)
    for t in range(x.shape[0]):
        for j in range(ids.shape[1]):
            e = ids[t, j]
            E = expert.swiglu_expert(x[t:t + 1], w1[e], w2[e])[0]
            assert abs(g["dgates"][t, j] - float(dy[t] @ E)) < 1e-12


def test_expert_subsets_add_up_to_the_full_gradient():
    x, ids, gates, w1, w2, dy = _case(5)
    full = backward.moe_backward(x, ids, gates, w1, w2, dy)
    a = backward.moe_backward(x, ids, gates, w1, w2, dy, experts=[0, 2])
    b = backward.moe_backward(x, ids, gates, w1, w2, dy, experts=[1, 3])
    np.testing.assert_array_equal(a["dw1"][0], full["dw1"][0])
    assert not a["dw1"][1].any() and not a["dw2"][3].any()
    np.testing.assert_allclose(a["dx"] + b["dx"], full["dx"], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(a["dgates"] + b["dgates"], full["dgates"], rtol=1e-13, atol=1e-14)
