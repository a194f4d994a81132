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


# ---- router gradient (d-logits through the softmax of Eq. 2) -------------------

_routing = routing


def _router_case(seed, T=20, Ne=10, k=3):
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((T, Ne))
    ids, _ = _routing.route_topk(z.astype(np.float32), k)
    dg = rng.standard_normal((T, k))
    return z, ids, dg


@pytest.mark.parametrize("renorm", [False, True])
def test_router_grad_finite_differences(renorm):
    z, ids, dg = _router_case(0)
    dz = backward.router_grad(z, ids, dg, renorm=renorm)

    def loss(zz):
        p = np.exp(zz - zz.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        g = np.take_along_axis(p, ids.astype(int), 1)
        if renorm:
            g = g / g.sum(1, keepdims=True)
        return float((dg * g).sum())

    h = 1e-6
    num = np.zeros_like(z)
    for t in range(z.shape[0]):
        for i in range(z.shape[1]):
            zp, zm = z.copy(), z.copy()
            zp[t, i] += h
            zm[t, i] -= h
            num[t, i] = (loss(zp) - loss(zm)) / (2 * h)
    np.testing.assert_allclose(dz, num, rtol=1e-6, atol=1e-9)


@pytest.mark.parametrize("renorm", [False, True])
def test_router_grad_matches_autograd(renorm):
    z, ids, dg = _router_case(1, T=64, Ne=16, k=4)
    zt = torch.tensor(z, dtype=torch.float64, requires_grad=True)
    g = torch.softmax(zt, dim=1).gather(1, torch.tensor(ids, dtype=torch.int64))
    if renorm:
        g = g / g.sum(1, keepdim=True)
    (g * torch.tensor(dg)).sum().backward()
    np.testing.assert_allclose(backward.router_grad(z, ids, dg, renorm=renorm),
                               zt.grad.numpy(), rtol=1e-11, atol=1e-14)


def test_router_grad_special_cases():
    z, ids, dg = _router_case(2, k=1)
    # one renormalised gate is the constant 1: no gradient
    assert not backward.router_grad(z, ids, dg, renorm=True).any()
    # all experts chosen: renormalisation changes nothing
    z, ids, dg = _router_case(3, Ne=6, k=6)
    np.testing.assert_allclose(backward.router_grad(z, ids, dg, renorm=True),
                               backward.router_grad(z, ids, dg, renorm=False), rtol=1e-12,
                               atol=1e-15)
    # the gradient of a softmax sums to zero over the logits of a token
    z, ids, dg = _router_case(4)
    for r in (False, True):
        np.testing.assert_allclose(backward.router_grad(z, ids, dg, renorm=r).sum(1), 0.0,
                                   atol=1e-14)
