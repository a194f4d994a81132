"""Host-side checks of the C ABI: the library builds, loads and exports every
entry point include/occult.h declares; argument checks reject bad calls before
anything is launched; the host placement (Algorithm 1) equals the oracle's.
No GPU is needed: nothing here launches a kernel."""
import ctypes
import os
import re

import numpy as np
import pytest

import synth
from oracle import coact, placement, routing

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def occ():
    from combine_top_route_gb300 import build
    build.build()
    import combine_top_route_gb300 as occ
    occ.lib()
    return occ


def declared_symbols():
    with open(os.path.join(ROOT, "include", "occult.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(occult_\w+)\s*\(", text, re.M)))


def test_exports_every_declared_symbol(occ):
    names = declared_symbols()
    assert len(names) >= 14
    L = ctypes.CDLL(occ.LIB_PATH)
    for n in names:
        assert hasattr(L, n), f"{n} is declared in occult.h but not exported"
    assert set(names) == set(occ.EXPORTED)


def declared_arity():
    """Number of parameters of every entry point declared in occult.h."""
    with open(os.path.join(ROOT, "include", "occult.h")) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    out = {}
    for m in re.finditer(r"^\s*(?:int|const char\*)\s+(occult_\w+)\s*\(([^;]*?)\)\s*;", text,
                         re.M | re.S):
        params = [p for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
        out[m.group(1)] = len(params)
    return out


def test_binding_constants_match_the_header(occ):
    """Every numeric #define of occult.h that the binding mirrors (as OCCULT_X or
    X) has the same value there; the ones the binding needs are all mirrored."""
    with open(os.path.join(ROOT, "include", "occult.h")) as f:
        text = f.read()
    defines = {m.group(1): int(m.group(2))
               for m in re.finditer(r"^#define OCCULT_(\w+)\s+(-?\d+)", text, re.M)}
    mirrored = {}
    for name, value in defines.items():
        for attr in ("OCCULT_" + name, name):
            if hasattr(occ, attr):
                mirrored[name] = getattr(occ, attr)
                break
    for name, value in mirrored.items():
        assert value == defines[name], f"OCCULT_{name}: header {defines[name]}, binding {value}"
    needed = {"F32", "BF16", "ERR_INVALID_ARG", "ERR_UNSUPPORTED", "ERR_WORKSPACE", "ERR_CUDA",
              "ERR_DEVICE_TIMEOUT", "ROUTE_EXACT", "ROUTE_DEVICE_LIMITED", "ROUTE_SCORE_PRUNED",
              "ROUTE_SIMILARITY_PRUNED", "MAX_EXPERTS", "MAX_VDEV", "MAX_TOPK", "MAX_SOURCES",
              "EPD_PAD", "WS_BUILD_BRIM", "WS_PROFILE_COACT", "WS_EXPERT_BWD",
              "STATIC_SCRATCH_BYTES"}
    assert needed <= set(mirrored), sorted(needed - set(mirrored))


def test_binding_signatures_match_the_header(occ):
    """Every ctypes prototype has as many arguments as its C declaration."""
    arity = declared_arity()
    assert set(arity) == set(occ.EXPORTED)
    for name, (_, args) in occ._SIGNATURES.items():
        assert len(args) == arity[name], f"{name}: binding {len(args)} args, header {arity[name]}"


def test_strerror(occ):
    assert occ.strerror(0) == "success"
    assert "timeout" in occ.strerror(occ.ERR_DEVICE_TIMEOUT) or "expired" in occ.strerror(occ.ERR_DEVICE_TIMEOUT)


def _desc(occ, **kw):
    ds = occ.desc_for(synth.CONFIGS["olmoe_fwd"])
    return ds.replace(**kw)


@pytest.mark.parametrize("kw,code", [
    (dict(n_vdev=7), -1),             # Ne % Nd != 0
    (dict(top_k=65), -1),             # k > Ne
    (dict(T=-1), -1),
    (dict(dtype=5), -1),
    (dict(route_mode=4), -1),
    (dict(route_mode=-1), -1),
    (dict(n_vdev=64), -2),            # more than 32 virtual devices
    (dict(top_k=17), -2),             # more than 16 experts per token
    (dict(d=2050), -2),               # bf16 rows must be multiples of 64
    (dict(inter=1000), -2),
    (dict(route_mode=1, limit_devices=0), -1),
    (dict(route_mode=1, limit_devices=1, top_k=9), -1),  # 1 device of 8 experts < k
    (dict(route_mode=2, limit_devices=0), -1),
    (dict(route_mode=2, limit_devices=1, top_k=9), -1),
    (dict(route_mode=3, limit_devices=9), -1),          # more than Nd devices
    (dict(n_shared=1, shared_inter=0), -1),
])
def test_bad_descriptors_are_rejected(occ, kw, code):
    assert occ.check_desc(_desc(occ, **kw)) == code


def test_calls_reject_bad_arguments_before_launching(occ):
    L = occ.lib()
    bad = _desc(occ, n_vdev=7)
    null = ctypes.c_void_p(0)
    assert L.occult_route(ctypes.byref(bad), null, null, null, null, null, null) == -1
    good = _desc(occ)
    # null pointers with a non-empty batch
    assert L.occult_route(ctypes.byref(good), null, null, null, null, null, null) == -1
    assert L.occult_build_brim(ctypes.byref(good), *([null] * 12), ctypes.c_size_t(0), null) == -1
    assert L.occult_dispatch(ctypes.byref(good), *([null] * 6)) == -1
    assert L.occult_expert_up(ctypes.byref(good), *([null] * 10)) == -1
    assert L.occult_expert_bwd(ctypes.byref(good), *([null] * 18), ctypes.c_size_t(0), null) == -1
    assert L.occult_gate_grad(ctypes.byref(good), *([null] * 9)) == -1
    assert L.occult_expert_down(ctypes.byref(good), *([null] * 6)) == -1
    assert L.occult_combine(ctypes.byref(good), *([null] * 9)) == -1
    assert L.occult_shared_ffn(ctypes.byref(good), *([null] * 8)) == -1   # no shared experts
    # a workspace smaller than the query is refused
    assert occ.workspace_size(good, occ.WS_BUILD_BRIM) > 0
    need = occ.workspace_size(good, occ.WS_PROFILE_COACT, 1024)
    assert need > 0
    assert L.occult_profile_coact(ctypes.byref(good), ctypes.c_void_p(16), 1024, null,
                                  ctypes.c_void_p(16), null, null, ctypes.c_void_p(16),
                                  ctypes.c_size_t(need - 1), null) == occ.ERR_WORKSPACE
    assert L.occult_place(null, 8, 4, null, null) == -1
    # the similarity mode needs its own entry point and its table, and the
    # table entry points their buffers
    sim = _desc(occ, route_mode=occ.ROUTE_SIMILARITY_PRUNED, limit_devices=2)
    v = ctypes.c_void_p(16)
    assert L.occult_route(ctypes.byref(sim), v, v, v, v, v, null) == -1
    assert L.occult_route_similarity(ctypes.byref(good), v, v, v, v, v, null, v, null) == -1
    assert L.occult_route_similarity(ctypes.byref(sim), v, v, null, v, v, null, v, null) == -1
    assert L.occult_similarity_accumulate(ctypes.byref(good), null, 16, v, null) == -1
    assert L.occult_similarity_accumulate(ctypes.byref(good), v, -1, v, null) == -1
    assert L.occult_similarity_finish(ctypes.byref(good), null, v, null) == -1
    assert L.occult_router_grad(ctypes.byref(good), v, null, v, v, null) == -1
    # the row-moving dispatches refuse rows that are not 16-byte aligned
    odd = ctypes.c_void_p(16 + 2)
    assert L.occult_dispatch(ctypes.byref(good), odd, v, v, v, null, null) == -1
    assert L.occult_dispatch(ctypes.byref(good), v, v, v, odd, null, null) == -1
    assert L.occult_dispatch_epd(ctypes.byref(good), odd, v, v, v, v, v, v, v, null) == -1
    assert L.occult_dispatch_epd(ctypes.byref(good), v, v, v, v, v, v, v, odd, null) == -1
    # stage-split merge and the sharded-source plan and exchange
    assert L.occult_merge_sfd(ctypes.byref(good), v, v, v, v, v, null, null) == -1
    assert L.occult_combine_sfd(ctypes.byref(good), v, null, null, v, null) == -1


def test_shard_entry_points_check_their_arguments(occ):
    L = occ.lib()
    good = _desc(occ)
    v = ctypes.c_void_p(256)
    null = ctypes.c_void_p(0)
    T = good.T

    def plan(off, n_src=None):
        host = (ctypes.c_int32 * len(off))(*off)
        n = len(off) - 1 if n_src is None else n_src
        return L.occult_shard_plan(ctypes.byref(good), n, ctypes.cast(host, ctypes.c_void_p),
                                   v, v, v, v, v, v, null)

    assert plan([0, T // 2, T // 4]) == -1            # not non-decreasing / does not end at T
    assert plan([1, T]) == -1                         # does not start at 0
    assert plan([0, T], n_src=0) == -1
    assert plan(list(range(0, 34)) + [T]) == -1       # more than 32 sources
    assert L.occult_shard_plan(ctypes.byref(good), 1, null, v, v, v, v, v, v, null) == -1

    def a2a(src, dst, row_bytes, reverse=0, n_src=2):
        return L.occult_all_to_all(ctypes.byref(good), n_src, v, v, v, ctypes.c_void_p(src),
                                   ctypes.c_void_p(dst), ctypes.c_int64(row_bytes), reverse, null)

    rows = T * min(good.top_k, good.n_vdev)
    rb = good.d * 2
    far = 1 << 40
    assert a2a(256, far, rb - 8) == -1                # row not a multiple of 16 bytes
    assert a2a(256, far, 0) == -1
    assert a2a(264, far, rb) == -1                    # unaligned source
    assert a2a(256, 256 + rows * rb - 16, rb) == -1   # overlapping buffers
    assert a2a(256, far, rb, reverse=2) == -1
    assert a2a(256, far, rb, n_src=33) == -1


def test_host_placement_matches_oracle(occ, golden):
    g = golden("placement_worked_example.json")
    L, e2v = occ.occult_place(np.array(g["C"]), g["n_vdev"])
    assert L.tolist() == g["expect"]["placement"]
    rng = np.random.default_rng(0)
    for Ne, Nd in [(8, 2), (16, 4), (64, 8), (60, 4), (6, 6), (64, 16)]:
        C = rng.integers(0, 40, size=(Ne, Ne))
        C = C + C.T
        L, e2v = occ.occult_place(C, Nd)
        want = placement.place(C, Nd)
        assert (L.numpy() == want).all()
        assert (e2v.numpy() == placement.expert_to_vdev(want)).all()


def test_host_placement_on_profiled_counts(occ):
    cfg = synth.CONFIGS["qwen_prefill"]
    ids, _ = routing.route_topk(synth.profiling_logits(cfg).numpy()[:4096], cfg.top_k)
    C = coact.coactivation(ids, cfg.n_experts)
    L, _ = occ.occult_place(C, cfg.n_vdev)
    assert (L.numpy() == placement.place(C, cfg.n_vdev)).all()


# entry points that take no layer descriptor first (checked by their own tests)
_NOT_DESC_FIRST = ("occult_strerror", "occult_check_desc", "occult_workspace_size",
                   "occult_device_error", "occult_selftest_wait", "occult_place",
                   "occult_zero_f32")


def test_zero_f32_refuses_bad_arguments(occ):
    """A null buffer with a non-zero length, or a negative length, is refused on
    the host."""
    L = occ.lib()
    assert L.occult_zero_f32(None, ctypes.c_int64(16), None) == occ.ERR_INVALID_ARG
    buf = (ctypes.c_float * 4)()
    assert L.occult_zero_f32(ctypes.cast(buf, ctypes.c_void_p), ctypes.c_int64(-1),
                             None) == occ.ERR_INVALID_ARG


def test_every_entry_point_refuses_null_buffers_before_launching(occ):
    """Every call taking a layer descriptor, given a valid non-empty layer and
    null buffers, returns OCCULT_ERR_INVALID_ARG: its arguments are checked on
    the host before anything launches (on this machine, without a GPU, a call
    that got past its checks would report a CUDA error instead)."""
    from combine_top_route_gb300 import _SIGNATURES
    L = occ.lib()
    good = _desc(occ)
    sim = _desc(occ, route_mode=occ.ROUTE_SIMILARITY_PRUNED, limit_devices=2)
    checked = []
    for name, (_, argtypes) in _SIGNATURES.items():
        if name in _NOT_DESC_FIRST:
            continue
        args = []
        for i, t in enumerate(argtypes):
            if i == 0:
                args.append(ctypes.byref(sim if name == "occult_route_similarity" else good))
            elif t is ctypes.c_void_p:
                args.append(ctypes.c_void_p(0))
            elif t is ctypes.c_int32 or t is ctypes.c_int:
                args.append(1)            # one source / one profiled token / a flag
            elif t is ctypes.c_int64:
                args.append(ctypes.c_int64(16))
            elif t is ctypes.c_size_t:
                args.append(ctypes.c_size_t(1 << 30))
            else:
                raise AssertionError(f"{name}: argument {i} of type {t}")
        rc = getattr(L, name)(*args)
        assert rc == occ.ERR_INVALID_ARG, f"{name} returned {rc}"
        checked.append(name)
    assert len(checked) >= 20


@pytest.mark.parametrize("bad", ["duplicate", "missing", "shape", "out_of_range"])
def test_layer_refuses_a_placement_that_is_not_a_partition(occ, bad):
    """The kernels index by the placement without checking it, so the binding
    refuses one that does not hold every expert exactly once (before any buffer
    is allocated: this runs on the CPU)."""
    import torch
    cfg = synth.CONFIGS["tiny_f32"]
    ds = occ.desc_for(cfg)
    L = np.arange(cfg.n_experts, dtype=np.int32).reshape(cfg.n_vdev, -1)
    if bad == "duplicate":
        L[0, 0] = L[0, 1]
    elif bad == "missing":
        L[1, 0] = L[0, 0]
    elif bad == "shape":
        L = L.reshape(-1)
    else:
        L[0, 0] = cfg.n_experts
    with pytest.raises(ValueError):
        occ.OccultMoE(ds, {}, torch.as_tensor(L), device="cpu")


def test_header_is_plain_c_and_links(occ, tmp_path):
    """occult.h compiles as C99 with warnings as errors, and a C program that
    takes the address of every declared entry point links against liboccult.so
    (nothing is run: the program would need a GPU)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = declared_symbols()
    src = tmp_path / "use_abi.c"
    src.write_text(
        '#include "occult.h"\n#include <stdio.h>\n'
        "int main(void) {\n"
        "  const void* fns[] = {\n"
        + "".join(f"    (const void*)&{n},\n" for n in names)
        + "  };\n"
        "  occult_desc_t d = {0};\n"
        "  printf(\"%d %d\\n\", (int)(sizeof fns / sizeof fns[0]), occult_check_desc(&d));\n"
        "  return 0;\n}\n")
    lib_dir = os.path.dirname(occ.LIB_PATH)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                        str(tmp_path / "use_abi"), "-L", lib_dir, "-loccult",
                        "-Wl,--allow-shlib-undefined"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
