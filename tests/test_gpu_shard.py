"""GPU parity of the sharded-source mode (the batch split over source devices,
the two all-to-alls real exchanges of row blocks) against the CPU oracle,
through the C ABI.

The plan (send map, block counts and offsets) and the exchanged rows are
compared bit for bit with the oracle's Algorithm 3 per source shard and its
block copies, on inputs the oracle computes itself.  The whole layer is checked
against Eq. 1 at the layer tolerance, and -- because the exchange only moves
rows -- bit for bit against the single-source path, forward and backward.
"""
import numpy as np
import pytest
import torch

import synth
from layer_cases import F32_EPS, assert_close_layer, expert_backward_bounds, make_case, \
    oracle_brims, reference_output, scatter_add_rows
from oracle import backward as obackward
from oracle import brim as obrim
from oracle import routing as orouting
from oracle import shard as oshard

pytestmark = pytest.mark.gpu

CFG = synth.CONFIGS


@pytest.fixture(scope="module")
def occ():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_top_route_gb300 import build
    build.build()
    import combine_top_route_gb300 as occ
    occ.lib()
    return occ


def i32(a):
    return torch.as_tensor(np.ascontiguousarray(np.asarray(a, np.int64).astype(np.int32))).cuda()


def vmask_of(act):
    bits = np.zeros(act.shape[0], dtype=np.int64)
    for d in range(act.shape[1]):
        bits |= act[:, d].astype(np.int64) << d
    return torch.as_tensor(bits.astype(np.uint32).view(np.int32)).cuda()


def splits(T, seed=0):
    """Equal shards, random cuts with empty shards, one source, 32 sources."""
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.integers(0, T + 1, size=6))
    return {
        "equal8": [s * T // 8 for s in range(9)],
        "random_with_empty": [0, int(cuts[0]), int(cuts[0]), *map(int, cuts[1:]), T, T],
        "one_source": [0, T],
        "sources32": [s * T // 32 for s in range(33)],
    }


CASES = {
    "olmoe_fwd": CFG["olmoe_fwd"],
    "ragged_1000": CFG["olmoe_fwd"].with_(name="ragged_1000", T=1000),
    "tiny_f32": CFG["tiny_f32"],
    "qwen_prefill": CFG["qwen_prefill"],
}


def oracle_setup(cfg, split):
    case = make_case(cfg, device="cpu", tensors=False)
    ids, gates, _ = case.oracle_route()
    act = orouting.token_devices(ids, case.e2v, cfg.n_vdev)
    b = oracle_brims(case, ids, gates)
    plan = oshard.shard_plan(act, split)
    return case, act, b, plan


def run_plan(occ, cfg, split, act, brim0):
    ds = occ.desc_for(cfg)
    n_src, Nd, T = len(split) - 1, cfg.n_vdev, cfg.T
    out = dict(brim0_send=torch.full((Nd, T), -7, dtype=torch.int32, device="cuda"),
               counts=torch.full((n_src, Nd), -7, dtype=torch.int32, device="cuda"),
               send_off=torch.full((n_src, Nd), -7, dtype=torch.int32, device="cuda"),
               recv_off=torch.full((n_src, Nd), -7, dtype=torch.int32, device="cuda"))
    occ.occult_shard_plan(ds, split, vmask_of(act), i32(brim0), **out)
    torch.cuda.synchronize()
    return ds, {n: v.cpu().numpy() for n, v in out.items()}


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("split_name", ["equal8", "random_with_empty", "one_source", "sources32"])
def test_shard_plan_bit_exact(occ, name, split_name):
    cfg = CASES[name]
    split = splits(cfg.T)[split_name]
    case, act, b, (b0s, counts, send_off, recv_off) = oracle_setup(cfg, split)
    _, got = run_plan(occ, cfg, split, act, b.brim0)
    assert (got["brim0_send"] == b0s).all()
    assert (got["counts"] == counts).all()
    assert (got["send_off"] == send_off).all()
    assert (got["recv_off"] == recv_off).all()


@pytest.mark.parametrize("name", ["olmoe_fwd", "ragged_1000", "tiny_f32"])
def test_all_to_all_moves_every_block(occ, name):
    """Both directions against the oracle's block copies, on bf16/fp32 rows and on
    fp32 stage-one rows; rows past N_sfd are left alone."""
    cfg = CASES[name]
    split = splits(cfg.T)["random_with_empty"]
    case, act, b, (b0s, counts, send_off, recv_off) = oracle_setup(cfg, split)
    ds = occ.desc_for(cfg)
    n_src = len(split) - 1
    n_max = cfg.T * min(cfg.top_k, cfg.n_vdev)
    n_sfd = b.n_sfd
    rng = np.random.default_rng(5)
    for dt in {cfg.torch_dtype, torch.float32}:
        send = np.zeros((n_max, cfg.d), np.float32)
        send[:n_sfd] = rng.standard_normal((n_sfd, cfg.d))
        send_t = torch.as_tensor(send).to(dt)
        send_h = send_t.float().numpy()
        want = oshard.all_to_all(send_h[:n_sfd], counts, send_off, recv_off)
        dst = torch.full((n_max, cfg.d), 7.0, dtype=dt, device="cuda")
        occ.occult_all_to_all(ds, n_src, i32(counts), i32(send_off), i32(recv_off),
                              send_t.cuda(), dst)
        torch.cuda.synchronize()
        got = dst.float().cpu().numpy()
        assert (got[:n_sfd] == want).all()
        assert (got[n_sfd:] == 7.0).all()
        back = torch.full((n_max, cfg.d), 7.0, dtype=dt, device="cuda")
        occ.occult_all_to_all(ds, n_src, i32(counts), i32(send_off), i32(recv_off), dst, back,
                              reverse=True)
        torch.cuda.synchronize()
        got = back.float().cpu().numpy()
        assert (got[:n_sfd] == oshard.all_to_all(want, counts, send_off, recv_off,
                                                 reverse=True)).all()
        assert (got[:n_sfd] == send_h[:n_sfd]).all()
        assert (got[n_sfd:] == 7.0).all()


def test_dispatch_then_exchange_reaches_the_receive_layout(occ):
    """Dispatch with the send map, then the first all-to-all: the receive buffers
    equal Algorithm 4's single-source SFD tensor."""
    cfg = CASES["olmoe_fwd"]
    split = splits(cfg.T)["equal8"]
    case = make_case(cfg)
    ids, gates, _ = case.oracle_route()
    act = orouting.token_devices(ids, case.e2v, cfg.n_vdev)
    b = oracle_brims(case, ids, gates)
    b0s, counts, send_off, recv_off = oshard.shard_plan(act, split)
    ds = occ.desc_for(cfg)
    n_max = cfg.T * min(cfg.top_k, cfg.n_vdev)
    x_send = torch.zeros(n_max, cfg.d, dtype=cfg.torch_dtype, device="cuda")
    x_recv = torch.zeros(n_max, cfg.d, dtype=cfg.torch_dtype, device="cuda")
    occ.occult_dispatch(ds, case.x, i32(b0s), vmask_of(act), x_send)
    occ.occult_all_to_all(ds, len(split) - 1, i32(counts), i32(send_off), i32(recv_off),
                          x_send, x_recv)
    torch.cuda.synchronize()
    x = case.host("x")
    assert (x_send[:b.n_sfd].float().cpu().numpy() == obrim.dispatch(x, b0s)).all()
    assert (x_recv[:b.n_sfd].float().cpu().numpy() == obrim.dispatch(x, b.brim0)).all()


def run_layer(occ, case, src_off=None, train=False, dy=None):
    moe = occ.OccultMoE(occ.desc_for(case.cfg), case.weights, torch.as_tensor(case.placement),
                        materialize_sfd=True, train=train, src_off=src_off)
    y = moe.forward(case.logits.cuda(), case.x).clone()
    grads = None
    if train:
        grads = [t.clone() for t in moe.backward(dy)] + [moe.dlogits.clone()]
    torch.cuda.synchronize()
    assert occ.device_error() == 0
    return moe, y, grads


@pytest.mark.parametrize("name", ["olmoe_fwd", "ragged_1000", "tiny_f32", "qwen_prefill"])
def test_sharded_layer(occ, name):
    """Eq. 1 at the layer tolerance; bit for bit the single-source output."""
    cfg = CASES[name]
    if name == "qwen_prefill":
        cfg = cfg.with_(T=2048)
    case = make_case(cfg)
    split = splits(cfg.T)["random_with_empty"]
    moe, y, _ = run_layer(occ, case, src_off=split)
    assert moe.launches_per_forward == 13 + (2 + int(cfg.shared_gate) if cfg.n_shared else 0)
    ids, gates, margin = case.oracle_route()
    toks = np.nonzero(margin > 1e-5)[0]
    assert_close_layer(y.cpu().numpy()[toks], reference_output(case, toks, ids, gates), cfg.dtype)
    _, y_single, _ = run_layer(occ, case)
    assert torch.equal(y, y_single)
    # the second exchange returned every stage-one row to its source's send layout
    act = orouting.token_devices(ids, case.e2v, cfg.n_vdev)
    b0s, counts, send_off, recv_off = oshard.shard_plan(act, split)
    n_sfd = int(counts.sum())
    y_sfd = moe.y_sfd[:n_sfd].cpu().numpy()
    assert (moe.y_send[:n_sfd].cpu().numpy() ==
            oshard.all_to_all(y_sfd, counts, send_off, recv_off, reverse=True)).all()


def test_sharded_training_step(occ):
    """Forward + backward with real exchanges: dx within its derived bound of the
    fp64 oracle, every output bit for bit the single-source step's."""
    cfg = synth.CONFIGS["olmoe_train"].with_(name="sharded_train", T=333, d=512, inter=192,
                                             n_vdev=8, n_src=4)
    case = make_case(cfg)
    dy = synth.upstream_grad(cfg, device="cuda")
    split = synth.source_offsets(cfg)
    moe, y, g_sh = run_layer(occ, case, src_off=split, train=True, dy=dy)
    assert moe.launches_per_backward == 12
    _, y1, g_single = run_layer(occ, case, train=True, dy=dy)
    assert torch.equal(y, y1)
    for a, b in zip(g_sh, g_single):
        assert torch.equal(a, b)
    ids, gates, _ = case.oracle_route()
    gates = gates.astype(np.float32).astype(np.float64)
    dy_h = dy.float().cpu().numpy()
    x, w1, w2 = case.host("x"), case.host("w1"), case.host("w2")
    ref = obackward.moe_backward(x, ids, gates, w1, w2, dy_h)
    T, k, d = cfg.T, cfg.top_k, cfg.d
    dx_b = np.zeros((T, d))
    dx_abs = np.zeros((T, d))
    for e in np.unique(ids):
        r, sl = np.nonzero(ids == e)
        bb = expert_backward_bounds(x[r], dy_h[r], w1[e], w2[e], gates[r, sl])
        scatter_add_rows(dx_b, r, bb["dx_rows_b"])
        scatter_add_rows(dx_abs, r, np.abs(bb["dx_rows"]) + bb["dx_rows_b"])
    dx_b += 2 * k * F32_EPS * dx_abs
    err = np.abs(g_sh[0].cpu().numpy().astype(np.float64) - ref["dx"])
    assert (err <= dx_b + 1e-30).all()
