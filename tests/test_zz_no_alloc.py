"""occult_build_brim_noalloc: the BRIM build for callers that cannot allocate.

Some callers cannot call cudaMalloc for a workspace (their device memory
belongs to an allocator they cannot reach, or their serving loop forbids
allocation after start-up).  The no-allocation entry point uses a static array
inside the library instead.  This file checks it, through the C ABI, against
occult_build_brim with a caller workspace, on two calls in a row (the second
one runs on the scratch the first one left behind).  It is collected last on
purpose, and it must pass both alone in a fresh process and after the rest of
the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from layer_cases import make_case

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


def _vmask(ids, e2v):
    bits = np.zeros(ids.shape[0], dtype=np.int64)
    for t in range(ids.shape[0]):
        for e in ids[t]:
            bits[t] |= 1 << int(e2v[e])
    return torch.as_tensor(bits.astype(np.uint32).view(np.int32)).cuda()


def _outputs(cfg, ds):
    T, k, Ne, Nd = cfg.T, cfg.top_k, cfg.n_experts, cfg.n_vdev
    i32 = dict(dtype=torch.int32, device="cuda")
    return dict(brim0=torch.full((Nd, T), -9, **i32), seg_off=torch.full((Nd + 1,), -9, **i32),
                brim1=torch.full((Ne, T), -9, **i32), exp_off=torch.full((Ne + 1,), -9, **i32),
                epd_src=torch.full((T * k,), -9, **i32),
                epd_gate=torch.full((T * k,), -9.0, dtype=torch.float32, device="cuda"),
                counts=torch.full((4,), -9, **i32))


@pytest.mark.parametrize("name,T", [("olmoe_fwd", 4096), ("qwen_prefill", 1000),
                                    ("tiny_f32", 256)])
def test_noalloc_matches_workspace_entry_point(occ, name, T):
    cfg = synth.CONFIGS[name].with_(T=T)
    case = make_case(cfg, device="cpu", tensors=False)
    ids, gates, _ = case.oracle_route()
    ds = occ.desc_for(cfg)
    ids_d = torch.as_tensor(ids.astype(np.int32)).cuda()
    gates_d = torch.as_tensor(gates.astype(np.float32)).cuda()
    vm = _vmask(ids, case.e2v)
    L = torch.as_tensor(case.placement.reshape(-1).astype(np.int32)).cuda()

    want = _outputs(cfg, ds)
    ws = torch.empty(max(1, occ.workspace_size(ds, occ.WS_BUILD_BRIM)), dtype=torch.uint8,
                     device="cuda")
    occ.occult_build_brim(ds, ids_d, gates_d, vm, L, ws=ws, **want)
    for call in range(2):
        got = _outputs(cfg, ds)
        occ.occult_build_brim_noalloc(ds, ids_d, gates_d, vm, L, **got)
        torch.cuda.synchronize()
        for n in want:
            # integer indices bit-exact; gates are copied, so exact as well
            assert torch.equal(got[n], want[n]), f"call {call}: {n} differs"
    assert occ.device_error() == 0


def test_noalloc_rejects_layers_beyond_its_scratch(occ):
    """A layer needing more scratch than the static array holds is refused on the host."""
    cfg = synth.CONFIGS["olmoe_fwd"].with_(T=70000, n_experts=256, n_vdev=8)
    ds = occ.desc_for(cfg)
    assert occ.workspace_size(ds, occ.WS_BUILD_BRIM) > occ.STATIC_SCRATCH_BYTES
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    ptrs = [ctypes.c_void_p(dummy.data_ptr())] * 11
    rc = occ.lib().occult_build_brim_noalloc(ctypes.byref(ds), *ptrs, None)
    assert rc == occ.ERR_WORKSPACE


def _ids_for(cfg, ds, occ):
    """Routed ids of the seeded batch (through occult_route: both entry points
    under test get the same ids, whatever they are) and the device masks."""
    case = make_case(cfg, device="cpu", tensors=False)
    T, k = cfg.T, cfg.top_k
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    gates = torch.empty(T, k, dtype=torch.float32, device="cuda")
    vmask = torch.empty(T, dtype=torch.int32, device="cuda")
    e2v = torch.as_tensor(case.e2v.astype(np.int32)).cuda()
    occ.occult_route(ds, case.logits.cuda(), e2v, ids, gates, vmask)
    L = torch.as_tensor(case.placement.reshape(-1).astype(np.int32)).cuda()
    return ids, gates, vmask, L


@pytest.mark.parametrize("T,Ne,Nd", [(32768, 256, 32), (97600, 64, 8)])
def test_noalloc_at_its_size_limit(occ, T, Ne, Nd):
    """The largest layers the static scratch holds (the two figures the header
    states) are accepted and equal the workspace entry point; one more token is
    refused with OCCULT_ERR_WORKSPACE before any launch."""
    cfg = synth.CONFIGS["olmoe_fwd"].with_(name=f"noalloc_{T}_{Ne}", T=T, n_experts=Ne,
                                           n_vdev=Nd, prof_tokens=4096)
    ds = occ.desc_for(cfg)
    assert occ.workspace_size(ds, occ.WS_BUILD_BRIM) <= occ.STATIC_SCRATCH_BYTES
    ids, gates, vmask, L = _ids_for(cfg, ds, occ)
    want = _outputs(cfg, ds)
    ws = torch.empty(occ.workspace_size(ds, occ.WS_BUILD_BRIM), dtype=torch.uint8, device="cuda")
    occ.occult_build_brim(ds, ids, gates, vmask, L, ws=ws, **want)
    got = _outputs(cfg, ds)
    occ.occult_build_brim_noalloc(ds, ids, gates, vmask, L, **got)
    torch.cuda.synchronize()
    for n in want:
        assert torch.equal(got[n], want[n]), f"{n} differs at T={T}, Ne={Ne}"

    over = cfg.with_(T=T + 1)
    ds1 = occ.desc_for(over)
    assert occ.workspace_size(ds1, occ.WS_BUILD_BRIM) > occ.STATIC_SCRATCH_BYTES
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    ptrs = [ctypes.c_void_p(dummy.data_ptr())] * 11
    assert occ.lib().occult_build_brim_noalloc(ctypes.byref(ds1), *ptrs, None) == occ.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert (dummy == 0).all()
    assert occ.device_error() == 0
