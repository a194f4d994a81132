"""Runtime properties of the C ABI on the GPU: failure detection (a bounded wait
that runs out latches an error and leaves the context usable) and CUDA-graph
capture of the layer's calls (the header promises both)."""
import numpy as np
import pytest
import torch

import synth
from layer_cases import assert_close_layer, make_case, reference_output

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def occ():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_top_route_gb300 import build
    build.build()
    import combine_top_route_gb300 as occ
    occ.lib()
    return occ


def small_case():
    cfg = synth.CONFIGS["olmoe_fwd"].with_(name="runtime", T=600, d=256, n_experts=16, top_k=4,
                                            inter=128, n_vdev=4, prof_tokens=2048)
    return make_case(cfg)


def test_bounded_wait_runs_out_and_the_context_survives(occ):
    assert occ.device_error() == 0
    # a barrier nothing completes: the wait gives up after 50 ms and latches the error
    occ.occult_selftest_wait(False, 50_000_000)
    torch.cuda.synchronize()
    assert occ.device_error() == occ.ERR_DEVICE_TIMEOUT
    assert occ.device_error() == 0          # reading clears it
    # the control: a completed barrier latches nothing
    occ.occult_selftest_wait(True, 50_000_000)
    torch.cuda.synchronize()
    assert occ.device_error() == 0
    # the context is still usable: a layer runs and meets Eq. 1
    case = small_case()
    moe = occ.OccultMoE(occ.desc_for(case.cfg), case.weights, torch.as_tensor(case.placement))
    y = moe.forward(case.logits.cuda(), case.x)
    torch.cuda.synchronize()
    toks = np.arange(case.cfg.T)
    assert_close_layer(y.cpu().numpy(), reference_output(case, toks), case.cfg.dtype)
    assert occ.device_error() == 0
    # out-of-range limits are refused before anything launches
    with pytest.raises(occ.OccultError):
        occ.occult_selftest_wait(False, 0)
    with pytest.raises(occ.OccultError):
        occ.occult_selftest_wait(False, 3_000_000_000)


@pytest.mark.parametrize("merge", ["ordered", "atomic"])
def test_forward_and_backward_replay_from_a_cuda_graph(occ, merge):
    """The whole forward (and the training backward) captured once and replayed on
    new inputs gives what eager calls give: bit for bit with the ordered merge,
    within the fp32 reordering of the atomic one."""
    case = small_case()
    cfg = case.cfg
    moe = occ.OccultMoE(occ.desc_for(cfg), case.weights, torch.as_tensor(case.placement),
                        train=True, merge=merge)
    logits = case.logits.cuda()
    x = case.x.clone()
    dy = synth.upstream_grad(cfg, device="cuda")
    # eager run (also the first calls, which set the library up before capture)
    moe.forward(logits, x)
    moe.backward(dy)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        moe.forward(logits, x)
        moe.backward(dy)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.forward(logits, x)
        moe.backward(dy)
    # new inputs in the captured buffers
    gen = torch.Generator(device="cuda").manual_seed(77)
    logits.copy_(torch.randn(logits.shape, generator=gen, device="cuda") * 2)
    x.copy_(torch.randn(x.shape, generator=gen, device="cuda").to(x.dtype))
    g.replay()
    torch.cuda.synchronize()
    got = [moe.y.clone(), moe.dx.clone(), moe.dw1.clone(), moe.dw2.clone(), moe.dgates.clone(),
           moe.dlogits.clone()]
    moe.forward(logits, x)
    moe.backward(dy)
    torch.cuda.synchronize()
    want = [moe.y, moe.dx, moe.dw1, moe.dw2, moe.dgates, moe.dlogits]
    for a, b, name in zip(got, want, ("y", "dx", "dw1", "dw2", "dgates", "dlogits")):
        if merge == "ordered" or name not in ("y", "dx"):
            assert torch.equal(a, b), name
        else:
            scale = float(b.abs().max())
            assert float((a - b).abs().max()) <= 1e-5 * scale, name
    assert occ.device_error() == 0


def kernel_nodes(fn):
    """Kernel launches of fn, counted as the kernel nodes of a CUDA graph capturing
    it (fn launches only this library's kernels)."""
    import ctypes
    try:
        g = torch.cuda.CUDAGraph(keep_graph=True)
    except TypeError:
        pytest.skip("this PyTorch cannot keep a captured graph")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    with torch.cuda.graph(g):
        fn()
    cu = ctypes.CDLL("libcuda.so.1")
    graph = ctypes.c_void_p(g.raw_cuda_graph())
    n = ctypes.c_size_t(0)
    assert cu.cuGraphGetNodes(graph, None, ctypes.byref(n)) == 0
    nodes = (ctypes.c_void_p * n.value)()
    assert cu.cuGraphGetNodes(graph, nodes, ctypes.byref(n)) == 0
    kinds = []
    for i in range(n.value):
        t = ctypes.c_int(-1)
        assert cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) == 0
        kinds.append(t.value)
    return sum(1 for t in kinds if t == 0)   # CU_GRAPH_NODE_TYPE_KERNEL


@pytest.mark.parametrize("merge,shared,train", [("atomic", False, True), ("ordered", False, True),
                                                ("atomic", True, False)])
def test_launch_counts_match_the_kernels_that_run(occ, merge, shared, train):
    """launches_per_forward / launches_per_backward (the bench's gpu_launches) equal
    the kernels a captured graph of the calls holds."""
    if shared:
        cfg = synth.CONFIGS["qwen_prefill"].with_(name="runtime_shared", T=600, d=256,
                                                   n_experts=16, top_k=4, inter=128, n_vdev=4,
                                                   shared_inter=256, prof_tokens=2048)
        case = make_case(cfg)
    else:
        case = small_case()
    moe = occ.OccultMoE(occ.desc_for(case.cfg), case.weights, torch.as_tensor(case.placement),
                        train=train, merge=merge)
    logits = case.logits.cuda()
    dy = synth.upstream_grad(case.cfg, device="cuda") if train else None
    moe.forward(logits, case.x)
    if train:
        moe.backward(dy)
    torch.cuda.synchronize()
    assert kernel_nodes(lambda: moe.forward(logits, case.x)) == moe.launches_per_forward
    if train:
        assert kernel_nodes(lambda: moe.backward(dy)) == moe.launches_per_backward
