"""The placement the bench's GPU arm uses comes from the library alone: the
profiling batch routed on the GPU, its co-activation counts (Eq. 3) on the GPU
and Algorithm 1 on the host, through the C ABI.  It equals the oracle's
Algorithm 1 on the oracle's routing of the same batch."""
import os
import sys

import pytest
import torch

import synth
from layer_cases import alg1_placement

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def occ():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_top_route_gb300 import build
    build.build()
    import combine_top_route_gb300 as occ
    occ.lib()
    return occ


@pytest.mark.parametrize("name", ["olmoe_fwd", "olmoe_train", "qwen_prefill", "deepseek_decode",
                                  "tiny_f32"])
def test_library_placement_equals_the_oracles(occ, name):
    sys.path.insert(0, ROOT)
    import bench
    cfg = synth.CONFIGS[name]
    L, offline = bench.library_placement(occ, cfg, torch.device("cuda", 0))
    assert (L.numpy() == alg1_placement(cfg)).all()
    assert offline["profiling_tokens"] == cfg.prof_tokens
    assert all(offline[k] >= 0 for k in ("route_ms", "profile_coact_ms", "place_ms"))
    assert occ.device_error() == 0
