"""Python binding of the Occult GB300 C ABI (``include/occult.h``).

Argument marshalling only: every function below has the name of a C entry
point, checks that the tensors it is handed are CUDA tensors of the expected
dtype and size, and passes their device pointers and the current CUDA stream to
``liboccult.so``.  Every step of the layer runs in the library's kernels; there
is no CPU or PyTorch fallback, and importing a function raises if the library
has not been built (``python -m combine_top_route_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "liboccult.so")

OCCULT_F32 = 0
OCCULT_BF16 = 1
ROUTE_EXACT = 0
ROUTE_DEVICE_LIMITED = 1
ROUTE_SCORE_PRUNED = 2
ROUTE_SIMILARITY_PRUNED = 3
MAX_EXPERTS = 256
MAX_VDEV = 32
MAX_TOPK = 16
MAX_SOURCES = 32

ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_WORKSPACE = -3
ERR_CUDA = -4
ERR_DEVICE_TIMEOUT = -5
WS_BUILD_BRIM = 0
WS_PROFILE_COACT = 1
WS_EXPERT_BWD = 2
STATIC_SCRATCH_BYTES = 1183744   # OCCULT_STATIC_SCRATCH_BYTES
EPD_PAD = 128                    # OCCULT_EPD_PAD


class occult_desc_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "T", "d", "n_experts", "top_k", "inter", "n_vdev", "dtype", "route_mode",
        "limit_devices", "renorm", "n_shared", "shared_inter", "shared_gate")]

    @property
    def n_loc(self) -> int:
        return self.n_experts // self.n_vdev

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == OCCULT_BF16 else torch.float32

    def replace(self, **kw) -> "occult_desc_t":
        out = occult_desc_t()
        for n, _ in self._fields_:
            setattr(out, n, kw.get(n, getattr(self, n)))
        return out


class OccultError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {code} ({strerror(code)})")
        self.code = code


_VP = ctypes.c_void_p
_I32 = ctypes.c_int32
_D = ctypes.POINTER(occult_desc_t)
_SIGNATURES = {
    "occult_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "occult_check_desc": (ctypes.c_int, [_D]),
    "occult_workspace_size": (ctypes.c_int, [_D, _I32, _I32, ctypes.POINTER(ctypes.c_size_t)]),
    "occult_device_error": (ctypes.c_int, [ctypes.POINTER(_I32)]),
    "occult_selftest_wait": (ctypes.c_int, [_I32, ctypes.c_int64, _VP]),
    "occult_place": (ctypes.c_int, [_VP, _I32, _I32, _VP, _VP]),
    "occult_route": (ctypes.c_int, [_D, _VP, _VP, _VP, _VP, _VP, _VP]),
    "occult_route_similarity": (ctypes.c_int, [_D] + [_VP] * 8),
    "occult_similarity_accumulate": (ctypes.c_int, [_D, _VP, _I32, _VP, _VP]),
    "occult_similarity_finish": (ctypes.c_int, [_D, _VP, _VP, _VP]),
    "occult_router_grad": (ctypes.c_int, [_D, _VP, _VP, _VP, _VP, _VP]),
    "occult_build_brim": (ctypes.c_int, [_D, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                         _VP, _VP, ctypes.c_size_t, _VP]),
    "occult_build_brim_noalloc": (ctypes.c_int, [_D, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                                 _VP, _VP, _VP, _VP]),
    "occult_dispatch": (ctypes.c_int, [_D, _VP, _VP, _VP, _VP, _VP, _VP]),
    "occult_dispatch_epd": (ctypes.c_int, [_D] + [_VP] * 9),
    "occult_expert_up": (ctypes.c_int, [_D] + [_VP] * 10),
    "occult_expert_down": (ctypes.c_int, [_D, _VP, _VP, _VP, _VP, _VP, _VP]),
    "occult_expert_down_merge": (ctypes.c_int, [_D] + [_VP] * 7 + [_I32, _VP]),
    "occult_expert_ffn": (ctypes.c_int, [_D, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                         _VP]),
    "occult_shared_ffn": (ctypes.c_int, [_D, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "occult_combine": (ctypes.c_int, [_D, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "occult_merge_sfd": (ctypes.c_int, [_D] + [_VP] * 7),
    "occult_combine_sfd": (ctypes.c_int, [_D] + [_VP] * 5),
    "occult_shard_plan": (ctypes.c_int, [_D, _I32] + [_VP] * 8),
    "occult_all_to_all": (ctypes.c_int, [_D, _I32, _VP, _VP, _VP, _VP, _VP, ctypes.c_int64,
                                         _I32, _VP]),
    "occult_expert_bwd": (ctypes.c_int, [_D] + [_VP] * 18 + [ctypes.c_size_t, _VP]),
    "occult_expert_bwd_merge": (ctypes.c_int, [_D] + [_VP] * 19 + [ctypes.c_size_t, _VP]),
    "occult_expert_dgrad_down": (ctypes.c_int, [_D] + [_VP] * 11 + [ctypes.c_size_t, _VP]),
    "occult_expert_dgrad_up": (ctypes.c_int, [_D] + [_VP] * 7 + [_I32, _VP]),
    "occult_expert_wgrad_down": (ctypes.c_int, [_D] + [_VP] * 8),
    "occult_expert_wgrad_up": (ctypes.c_int, [_D] + [_VP] * 8),
    "occult_zero_f32": (ctypes.c_int, [_VP, ctypes.c_int64, _VP]),
    "occult_gate_grad": (ctypes.c_int, [_D] + [_VP] * 9),
    "occult_profile_coact": (ctypes.c_int, [_D, _VP, _I32, _VP, _VP, _VP, _VP, _VP,
                                            ctypes.c_size_t, _VP]),
}
EXPORTED = tuple(_SIGNATURES)

_lib_handle = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m combine_top_route_gb300.build`")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            f = getattr(h, name)
            f.restype = res
            f.argtypes = args
        _lib_handle = h
    return _lib_handle


def strerror(code: int) -> str:
    return lib().occult_strerror(code).decode()


def _call(name: str, *args) -> None:
    rc = getattr(lib(), name)(*args)
    if rc != 0:
        raise OccultError(name, rc)


def _dev(t: Optional[torch.Tensor], dtype: Optional[torch.dtype] = None, numel: Optional[int] = None,
         name: str = "tensor", nullable: bool = False):
    """Device pointer of a contiguous CUDA tensor (checked), or None."""
    if t is None:
        if nullable:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs {numel}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def epd_copy_rows(desc: occult_desc_t) -> int:
    """Rows of a padded EPD copy (x_epd, dy_epd): expert e's rows start at
    exp_off[e] + EPD_PAD * e, zeros after them to the next multiple of EPD_PAD."""
    return desc.T * desc.top_k + EPD_PAD * desc.n_experts


def check_desc(desc: occult_desc_t) -> int:
    return lib().occult_check_desc(ctypes.byref(desc))


def device_error() -> int:
    code = _I32(0)
    _call("occult_device_error", ctypes.byref(code))
    return code.value


def workspace_size(desc: occult_desc_t, op: int, n_tok: int = 0) -> int:
    """Device workspace bytes of the entry point selected by `op` (WS_* constants)."""
    n = ctypes.c_size_t(0)
    _call("occult_workspace_size", ctypes.byref(desc), op, n_tok, ctypes.byref(n))
    return n.value


def occult_selftest_wait(complete: bool, limit_ns: int, stream=None) -> None:
    """One bounded device wait that gives up (complete=False) or completes (see occult.h)."""
    _call("occult_selftest_wait", int(bool(complete)), ctypes.c_int64(int(limit_ns)),
          _stream(stream))


def occult_place(C, n_vdev: int):
    """Algorithm 1 on host counts C [Ne, Ne] (int64, CPU).  Returns (placement, expert_to_vdev)."""
    C = torch.as_tensor(C, dtype=torch.int64).contiguous()
    Ne = C.shape[0]
    placement = torch.empty(n_vdev, Ne // n_vdev, dtype=torch.int32)
    e2v = torch.empty(Ne, dtype=torch.int32)
    _call("occult_place", ctypes.c_void_p(C.data_ptr()), Ne, n_vdev,
          ctypes.c_void_p(placement.data_ptr()), ctypes.c_void_p(e2v.data_ptr()))
    return placement, e2v


def occult_route(desc, logits, expert_to_vdev, ids, gates, vmask, stream=None):
    T, Ne, k = desc.T, desc.n_experts, desc.top_k
    _call("occult_route", ctypes.byref(desc), _dev(logits, torch.float32, T * Ne, "logits"),
          _dev(expert_to_vdev, torch.int32, Ne, "expert_to_vdev"),
          _dev(ids, torch.int32, T * k, "ids"), _dev(gates, torch.float32, T * k, "gates"),
          _dev(vmask, torch.int32, T, "vmask"), _stream(stream))


def occult_route_similarity(desc, logits, expert_to_vdev, table, ids, gates, vmask, routed=None,
                            stream=None):
    T, Ne, k = desc.T, desc.n_experts, desc.top_k
    _call("occult_route_similarity", ctypes.byref(desc),
          _dev(logits, torch.float32, T * Ne, "logits"),
          _dev(expert_to_vdev, torch.int32, Ne, "expert_to_vdev"),
          _dev(table, torch.float32, Ne * Ne, "table"),
          _dev(ids, torch.int32, T * k, "ids"), _dev(gates, torch.float32, T * k, "gates"),
          _dev(routed, torch.int32, T * k, "routed", nullable=True),
          _dev(vmask, torch.int32, T, "vmask"), _stream(stream))


def occult_similarity_accumulate(desc, logits, n_tok, G, stream=None):
    Ne = desc.n_experts
    _call("occult_similarity_accumulate", ctypes.byref(desc),
          _dev(logits, torch.float32, n_tok * Ne, "logits", nullable=n_tok == 0), n_tok,
          _dev(G, torch.float64, Ne * Ne, "G"), _stream(stream))


def occult_similarity_finish(desc, G, table, stream=None):
    Ne = desc.n_experts
    _call("occult_similarity_finish", ctypes.byref(desc), _dev(G, torch.float64, Ne * Ne, "G"),
          _dev(table, torch.float32, Ne * Ne, "table"), _stream(stream))


def occult_router_grad(desc, logits, gate_ids, dgates, dlogits, stream=None):
    T, Ne, k = desc.T, desc.n_experts, desc.top_k
    _call("occult_router_grad", ctypes.byref(desc), _dev(logits, torch.float32, T * Ne, "logits"),
          _dev(gate_ids, torch.int32, T * k, "gate_ids"),
          _dev(dgates, torch.float32, T * k, "dgates"),
          _dev(dlogits, torch.float32, T * Ne, "dlogits"), _stream(stream))


def occult_build_brim(desc, ids, gates, vmask, placement, brim0, seg_off, brim1, exp_off,
                      epd_src, epd_gate, counts, ws, stream=None):
    T, Ne, k, Nd = desc.T, desc.n_experts, desc.top_k, desc.n_vdev
    i32, f32 = torch.int32, torch.float32
    need = workspace_size(desc, WS_BUILD_BRIM)
    _call("occult_build_brim", ctypes.byref(desc), _dev(ids, i32, T * k, "ids"),
          _dev(gates, f32, T * k, "gates"), _dev(vmask, i32, T, "vmask"),
          _dev(placement, i32, Ne, "placement"), _dev(brim0, i32, Nd * T, "brim0"),
          _dev(seg_off, i32, Nd + 1, "seg_off"), _dev(brim1, i32, Ne * T, "brim1"),
          _dev(exp_off, i32, Ne + 1, "exp_off"), _dev(epd_src, i32, T * k, "epd_src"),
          _dev(epd_gate, f32, T * k, "epd_gate"), _dev(counts, i32, 4, "counts"),
          _dev(ws, torch.uint8, need, "ws", nullable=need == 0), ctypes.c_size_t(need),
          _stream(stream))


def occult_build_brim_noalloc(desc, ids, gates, vmask, placement, brim0, seg_off, brim1,
                              exp_off, epd_src, epd_gate, counts, stream=None):
    """occult_build_brim with the library's static scratch instead of a workspace.

    For callers that cannot allocate device memory; see include/occult.h.
    Calls that overlap on the GPU share the scratch and race.
    """
    T, Ne, k, Nd = desc.T, desc.n_experts, desc.top_k, desc.n_vdev
    i32, f32 = torch.int32, torch.float32
    _call("occult_build_brim_noalloc", ctypes.byref(desc), _dev(ids, i32, T * k, "ids"),
          _dev(gates, f32, T * k, "gates"), _dev(vmask, i32, T, "vmask"),
          _dev(placement, i32, Ne, "placement"), _dev(brim0, i32, Nd * T, "brim0"),
          _dev(seg_off, i32, Nd + 1, "seg_off"), _dev(brim1, i32, Ne * T, "brim1"),
          _dev(exp_off, i32, Ne + 1, "exp_off"), _dev(epd_src, i32, T * k, "epd_src"),
          _dev(epd_gate, f32, T * k, "epd_gate"), _dev(counts, i32, 4, "counts"),
          _stream(stream))


def occult_dispatch(desc, x, brim0, vmask, x_sfd, sfd_tok=None, stream=None):
    T, d, Nd = desc.T, desc.d, desc.n_vdev
    dt = desc.torch_dtype
    n_sfd_max = T * min(desc.top_k, Nd)
    _call("occult_dispatch", ctypes.byref(desc), _dev(x, dt, T * d, "x"),
          _dev(brim0, torch.int32, Nd * T, "brim0"), _dev(vmask, torch.int32, T, "vmask"),
          _dev(x_sfd, dt, n_sfd_max * d, "x_sfd"),
          _dev(sfd_tok, torch.int32, n_sfd_max, "sfd_tok", nullable=True), _stream(stream))


def occult_dispatch_epd(desc, x, ids, placement, brim0, seg_off, brim1, exp_off, x_epd,
                        stream=None):
    """Token rows straight to the padded EPD layout (one source; see occult.h)."""
    T, d, Ne, k, Nd = desc.T, desc.d, desc.n_experts, desc.top_k, desc.n_vdev
    i32 = torch.int32
    _call("occult_dispatch_epd", ctypes.byref(desc), _dev(x, desc.torch_dtype, T * d, "x"),
          _dev(ids, i32, T * k, "ids"), _dev(placement, i32, Ne, "placement"),
          _dev(brim0, i32, Nd * T, "brim0"), _dev(seg_off, i32, Nd + 1, "seg_off"),
          _dev(brim1, i32, Ne * T, "brim1"), _dev(exp_off, i32, Ne + 1, "exp_off"),
          _dev(x_epd, desc.torch_dtype, epd_copy_rows(desc) * d, "x_epd"), _stream(stream))


def occult_expert_up(desc, x_sfd, epd_src, epd_gate, exp_off, placement, w1, h_epd, gu_epd=None,
                     x_epd=None, stream=None):
    """h' (and, training, G|U and the padded EPD copy x_epd of the gathered rows)."""
    T, d, Ne, k, I = desc.T, desc.d, desc.n_experts, desc.top_k, desc.inter
    dt = desc.torch_dtype
    _call("occult_expert_up", ctypes.byref(desc),
          _dev(x_sfd, dt, T * min(k, desc.n_vdev) * d, "x_sfd"),
          _dev(epd_src, torch.int32, T * k, "epd_src"),
          _dev(epd_gate, torch.float32, T * k, "epd_gate"),
          _dev(exp_off, torch.int32, Ne + 1, "exp_off"),
          _dev(placement, torch.int32, Ne, "placement"),
          _dev(w1, dt, Ne * 2 * I * d, "w1"), _dev(h_epd, dt, T * k * I, "h_epd"),
          _dev(gu_epd, dt, T * k * 2 * I, "gu_epd", nullable=True),
          _dev(x_epd, dt, epd_copy_rows(desc) * d, "x_epd", nullable=True), _stream(stream))


def occult_expert_bwd(desc, x_sfd, dy_sfd, epd_src, epd_gate, exp_off, placement, w1, w2, h_epd,
                      gu_epd, dgu_epd, dx_epd, dw1, dw2, dg_epd, ws, x_epd=None, dy_epd=None,
                      stream=None):
    T, d, Ne, k, I = desc.T, desc.d, desc.n_experts, desc.top_k, desc.inter
    dt, f32, i32 = desc.torch_dtype, torch.float32, torch.int32
    n_sfd_max = T * min(k, desc.n_vdev)
    need = workspace_size(desc, WS_EXPERT_BWD)
    _call("occult_expert_bwd", ctypes.byref(desc),
          _dev(x_sfd, dt, n_sfd_max * d, "x_sfd", nullable=x_epd is not None),
          _dev(dy_sfd, dt, n_sfd_max * d, "dy_sfd", nullable=dy_epd is not None),
          _dev(epd_src, i32, T * k, "epd_src"),
          _dev(epd_gate, f32, T * k, "epd_gate"), _dev(exp_off, i32, Ne + 1, "exp_off"),
          _dev(placement, i32, Ne, "placement"), _dev(w1, dt, Ne * 2 * I * d, "w1"),
          _dev(w2, dt, Ne * d * I, "w2"), _dev(h_epd, dt, T * k * I, "h_epd"),
          _dev(gu_epd, dt, T * k * 2 * I, "gu_epd"), _dev(dgu_epd, dt, T * k * 2 * I, "dgu_epd"),
          _dev(dx_epd, f32, T * k * d, "dx_epd"), _dev(dw1, f32, Ne * 2 * I * d, "dw1"),
          _dev(dw2, f32, Ne * d * I, "dw2"), _dev(dg_epd, f32, T * k, "dg_epd"),
          _dev(x_epd, dt, epd_copy_rows(desc) * d, "x_epd", nullable=True),
          _dev(dy_epd, dt, epd_copy_rows(desc) * d, "dy_epd", nullable=True),
          _dev(ws, torch.uint8, need, "ws", nullable=need == 0), ctypes.c_size_t(need),
          _stream(stream))


def occult_expert_bwd_merge(desc, x_sfd, dy_sfd, epd_src, epd_gate, exp_off, placement, w1, w2,
                            h_epd, gu_epd, dgu_epd, sfd_tok, dx, dw1, dw2, dg_epd, ws,
                            x_epd=None, dy_epd=None, stream=None):
    """occult_expert_bwd with dx merged by fp32 atomics into the token rows (occult.h)."""
    T, d, Ne, k, I = desc.T, desc.d, desc.n_experts, desc.top_k, desc.inter
    dt, f32, i32 = desc.torch_dtype, torch.float32, torch.int32
    n_sfd_max = T * min(k, desc.n_vdev)
    need = workspace_size(desc, WS_EXPERT_BWD)
    _call("occult_expert_bwd_merge", ctypes.byref(desc),
          _dev(x_sfd, dt, n_sfd_max * d, "x_sfd", nullable=x_epd is not None),
          _dev(dy_sfd, dt, n_sfd_max * d, "dy_sfd", nullable=dy_epd is not None),
          _dev(epd_src, i32, T * k, "epd_src"),
          _dev(epd_gate, f32, T * k, "epd_gate"), _dev(exp_off, i32, Ne + 1, "exp_off"),
          _dev(placement, i32, Ne, "placement"), _dev(w1, dt, Ne * 2 * I * d, "w1"),
          _dev(w2, dt, Ne * d * I, "w2"), _dev(h_epd, dt, T * k * I, "h_epd"),
          _dev(gu_epd, dt, T * k * 2 * I, "gu_epd"), _dev(dgu_epd, dt, T * k * 2 * I, "dgu_epd"),
          _dev(sfd_tok, i32, n_sfd_max, "sfd_tok"), _dev(dx, f32, T * d, "dx"),
          _dev(dw1, f32, Ne * 2 * I * d, "dw1"), _dev(dw2, f32, Ne * d * I, "dw2"),
          _dev(dg_epd, f32, T * k, "dg_epd"),
          _dev(x_epd, dt, epd_copy_rows(desc) * d, "x_epd", nullable=True),
          _dev(dy_epd, dt, epd_copy_rows(desc) * d, "dy_epd", nullable=True),
          _dev(ws, torch.uint8, need, "ws", nullable=need == 0), ctypes.c_size_t(need),
          _stream(stream))


def occult_expert_dgrad_down(desc, dy_sfd, epd_src, epd_gate, exp_off, placement, w2, gu_epd,
                             dgu_epd, dg_epd, ws, dy_epd=None, stream=None):
    """dh', dG|dU and dg; dy rows gathered from dy_sfd (then copied to dy_epd when
    given), or, with dy_sfd None, read from dy's padded EPD rows dy_epd."""
    T, d, Ne, k, I = desc.T, desc.d, desc.n_experts, desc.top_k, desc.inter
    dt, f32, i32 = desc.torch_dtype, torch.float32, torch.int32
    need = workspace_size(desc, WS_EXPERT_BWD)
    _call("occult_expert_dgrad_down", ctypes.byref(desc),
          _dev(dy_sfd, dt, T * min(k, desc.n_vdev) * d, "dy_sfd", nullable=dy_epd is not None),
          _dev(epd_src, i32, T * k, "epd_src"), _dev(epd_gate, f32, T * k, "epd_gate"),
          _dev(exp_off, i32, Ne + 1, "exp_off"), _dev(placement, i32, Ne, "placement"),
          _dev(w2, dt, Ne * d * I, "w2"), _dev(gu_epd, dt, T * k * 2 * I, "gu_epd"),
          _dev(dgu_epd, dt, T * k * 2 * I, "dgu_epd"), _dev(dg_epd, f32, T * k, "dg_epd"),
          _dev(dy_epd, dt, epd_copy_rows(desc) * d, "dy_epd", nullable=True),
          _dev(ws, torch.uint8, need, "ws", nullable=need == 0), ctypes.c_size_t(need),
          _stream(stream))


def occult_expert_dgrad_up(desc, dgu_epd, epd_src, exp_off, placement, w1, dx, sfd_tok=None,
                           zero_dx=False, stream=None):
    """dx rows of the backward; merged into dx [T, d] when sfd_tok is given (occult.h)."""
    T, d, Ne, k, I = desc.T, desc.d, desc.n_experts, desc.top_k, desc.inter
    dt, i32 = desc.torch_dtype, torch.int32
    _call("occult_expert_dgrad_up", ctypes.byref(desc),
          _dev(dgu_epd, dt, T * k * 2 * I, "dgu_epd"), _dev(epd_src, i32, T * k, "epd_src"),
          _dev(exp_off, i32, Ne + 1, "exp_off"), _dev(placement, i32, Ne, "placement"),
          _dev(w1, dt, Ne * 2 * I * d, "w1"),
          _dev(sfd_tok, i32, T * min(k, desc.n_vdev), "sfd_tok", nullable=True),
          _dev(dx, torch.float32, (T if sfd_tok is not None else T * k) * d, "dx"),
          int(bool(zero_dx)), _stream(stream))


def occult_expert_wgrad_down(desc, dy_sfd, epd_src, exp_off, placement, h_epd, dw2, dy_epd=None,
                             stream=None):
    """dW2; the dy rows gathered from dy_sfd, or read from their padded EPD copy dy_epd."""
    T, d, Ne, k, I = desc.T, desc.d, desc.n_experts, desc.top_k, desc.inter
    dt, i32 = desc.torch_dtype, torch.int32
    tiles = dy_epd is not None
    _call("occult_expert_wgrad_down", ctypes.byref(desc),
          _dev(dy_sfd, dt, T * min(k, desc.n_vdev) * d, "dy_sfd", nullable=tiles),
          _dev(epd_src, i32, T * k, "epd_src", nullable=tiles),
          _dev(dy_epd, dt, epd_copy_rows(desc) * d, "dy_epd", nullable=True),
          _dev(exp_off, i32, Ne + 1, "exp_off"),
          _dev(placement, i32, Ne, "placement"), _dev(h_epd, dt, T * k * I, "h_epd"),
          _dev(dw2, torch.float32, Ne * d * I, "dw2"), _stream(stream))


def occult_expert_wgrad_up(desc, x_sfd, epd_src, exp_off, placement, dgu_epd, dw1, x_epd=None,
                           stream=None):
    """dW1; the x rows gathered from x_sfd, or read from their padded EPD copy x_epd."""
    T, d, Ne, k, I = desc.T, desc.d, desc.n_experts, desc.top_k, desc.inter
    dt, i32 = desc.torch_dtype, torch.int32
    tiles = x_epd is not None
    _call("occult_expert_wgrad_up", ctypes.byref(desc),
          _dev(x_sfd, dt, T * min(k, desc.n_vdev) * d, "x_sfd", nullable=tiles),
          _dev(epd_src, i32, T * k, "epd_src", nullable=tiles),
          _dev(x_epd, dt, epd_copy_rows(desc) * d, "x_epd", nullable=True),
          _dev(exp_off, i32, Ne + 1, "exp_off"),
          _dev(placement, i32, Ne, "placement"), _dev(dgu_epd, dt, T * k * 2 * I, "dgu_epd"),
          _dev(dw1, torch.float32, Ne * 2 * I * d, "dw1"), _stream(stream))


def occult_zero_f32(buf, stream=None):
    """buf (fp32, contiguous, on the device) = 0."""
    _call("occult_zero_f32", _dev(buf, torch.float32, buf.numel(), "buf"),
          ctypes.c_int64(buf.numel()), _stream(stream))


def occult_gate_grad(desc, ids, placement, brim0, seg_off, brim1, exp_off, dg_epd, dgates,
                     stream=None):
    T, Ne, k, Nd = desc.T, desc.n_experts, desc.top_k, desc.n_vdev
    i32, f32 = torch.int32, torch.float32
    _call("occult_gate_grad", ctypes.byref(desc), _dev(ids, i32, T * k, "ids"),
          _dev(placement, i32, Ne, "placement"), _dev(brim0, i32, Nd * T, "brim0"),
          _dev(seg_off, i32, Nd + 1, "seg_off"), _dev(brim1, i32, Ne * T, "brim1"),
          _dev(exp_off, i32, Ne + 1, "exp_off"), _dev(dg_epd, f32, T * k, "dg_epd"),
          _dev(dgates, f32, T * k, "dgates"), _stream(stream))


def occult_expert_down(desc, h_epd, exp_off, placement, w2, y_epd, stream=None):
    T, d, Ne, k, I = desc.T, desc.d, desc.n_experts, desc.top_k, desc.inter
    dt = desc.torch_dtype
    _call("occult_expert_down", ctypes.byref(desc), _dev(h_epd, dt, T * k * I, "h_epd"),
          _dev(exp_off, torch.int32, Ne + 1, "exp_off"),
          _dev(placement, torch.int32, Ne, "placement"), _dev(w2, dt, Ne * d * I, "w2"),
          _dev(y_epd, torch.float32, T * k * d, "y_epd"), _stream(stream))


def occult_expert_down_merge(desc, h_epd, exp_off, placement, w2, epd_src, sfd_tok, y,
                             zero_y=True, stream=None):
    """The down-projection with the merge as fp32 atomic adds into y (see occult.h)."""
    T, d, Ne, k, I, Nd = desc.T, desc.d, desc.n_experts, desc.top_k, desc.inter, desc.n_vdev
    dt, i32 = desc.torch_dtype, torch.int32
    _call("occult_expert_down_merge", ctypes.byref(desc), _dev(h_epd, dt, T * k * I, "h_epd"),
          _dev(exp_off, i32, Ne + 1, "exp_off"), _dev(placement, i32, Ne, "placement"),
          _dev(w2, dt, Ne * d * I, "w2"), _dev(epd_src, i32, T * k, "epd_src"),
          _dev(sfd_tok, i32, T * min(k, Nd), "sfd_tok"), _dev(y, torch.float32, T * d, "y"),
          int(bool(zero_y)), _stream(stream))


def occult_expert_ffn(desc, x_sfd, epd_src, epd_gate, exp_off, placement, w1, w2, h_epd, y_epd,
                      stream=None):
    T, d, Ne, k, I = desc.T, desc.d, desc.n_experts, desc.top_k, desc.inter
    dt = desc.torch_dtype
    _call("occult_expert_ffn", ctypes.byref(desc),
          _dev(x_sfd, dt, T * min(k, desc.n_vdev) * d, "x_sfd"),
          _dev(epd_src, torch.int32, T * k, "epd_src"),
          _dev(epd_gate, torch.float32, T * k, "epd_gate"),
          _dev(exp_off, torch.int32, Ne + 1, "exp_off"),
          _dev(placement, torch.int32, Ne, "placement"), _dev(w1, dt, Ne * 2 * I * d, "w1"),
          _dev(w2, dt, Ne * d * I, "w2"), _dev(h_epd, dt, T * k * I, "h_epd"),
          _dev(y_epd, torch.float32, T * k * d, "y_epd"), _stream(stream))


def occult_shared_ffn(desc, x, ws1, ws2, w_sg, h_s, s_gate, y_s, stream=None):
    T, d = desc.T, desc.d
    S = desc.n_shared * desc.shared_inter
    dt = desc.torch_dtype
    _call("occult_shared_ffn", ctypes.byref(desc), _dev(x, dt, T * d, "x"),
          _dev(ws1, dt, 2 * S * d, "ws1"), _dev(ws2, dt, d * S, "ws2"),
          _dev(w_sg, dt, d, "w_sg", nullable=not desc.shared_gate),
          _dev(h_s, dt, T * S, "h_s"),
          _dev(s_gate, torch.float32, T, "s_gate", nullable=not desc.shared_gate),
          _dev(y_s, torch.float32, T * d, "y_s"), _stream(stream))


def occult_combine(desc, y_epd, brim0, seg_off, brim1, exp_off, y, y_shared=None, y_sfd=None,
                   stream=None):
    T, d, Ne, k, Nd = desc.T, desc.d, desc.n_experts, desc.top_k, desc.n_vdev
    f32 = torch.float32
    i32 = torch.int32
    _call("occult_combine", ctypes.byref(desc), _dev(y_epd, f32, T * k * d, "y_epd"),
          _dev(brim0, i32, Nd * T, "brim0"), _dev(seg_off, i32, Nd + 1, "seg_off"),
          _dev(brim1, i32, Ne * T, "brim1"), _dev(exp_off, i32, Ne + 1, "exp_off"),
          _dev(y_shared, f32, T * d, "y_shared", nullable=True),
          _dev(y_sfd, f32, T * min(k, Nd) * d, "y_sfd", nullable=True),
          _dev(y, f32, T * d, "y"), _stream(stream))


def occult_merge_sfd(desc, y_epd, brim0, seg_off, brim1, exp_off, y_sfd, stream=None):
    T, d, Ne, k, Nd = desc.T, desc.d, desc.n_experts, desc.top_k, desc.n_vdev
    f32, i32 = torch.float32, torch.int32
    _call("occult_merge_sfd", ctypes.byref(desc), _dev(y_epd, f32, T * k * d, "y_epd"),
          _dev(brim0, i32, Nd * T, "brim0"), _dev(seg_off, i32, Nd + 1, "seg_off"),
          _dev(brim1, i32, Ne * T, "brim1"), _dev(exp_off, i32, Ne + 1, "exp_off"),
          _dev(y_sfd, f32, T * min(k, Nd) * d, "y_sfd"), _stream(stream))


def occult_combine_sfd(desc, y_sfd, row_map, y, y_shared=None, stream=None):
    T, d, k, Nd = desc.T, desc.d, desc.top_k, desc.n_vdev
    f32 = torch.float32
    _call("occult_combine_sfd", ctypes.byref(desc),
          _dev(y_sfd, f32, T * min(k, Nd) * d, "y_sfd"),
          _dev(row_map, torch.int32, Nd * T, "row_map"),
          _dev(y_shared, f32, T * d, "y_shared", nullable=True), _dev(y, f32, T * d, "y"),
          _stream(stream))


def occult_shard_plan(desc, src_off, vmask, brim0, brim0_send, counts, send_off, recv_off,
                      stream=None):
    """``src_off``: host sequence of n_src + 1 token offsets of the source shards."""
    T, Nd = desc.T, desc.n_vdev
    off = [int(v) for v in src_off]
    n_src = len(off) - 1
    host = (ctypes.c_int32 * len(off))(*off)
    i32 = torch.int32
    _call("occult_shard_plan", ctypes.byref(desc), n_src, ctypes.cast(host, ctypes.c_void_p),
          _dev(vmask, i32, T, "vmask"), _dev(brim0, i32, Nd * T, "brim0"),
          _dev(brim0_send, i32, Nd * T, "brim0_send"),
          _dev(counts, i32, max(n_src, 1) * Nd, "counts"),
          _dev(send_off, i32, max(n_src, 1) * Nd, "send_off"),
          _dev(recv_off, i32, max(n_src, 1) * Nd, "recv_off"), _stream(stream))


def occult_all_to_all(desc, n_src, counts, send_off, recv_off, src, dst, reverse=False,
                      stream=None):
    """Row blocks between the send and receive layouts; the row size is src's last dim."""
    T, Nd = desc.T, desc.n_vdev
    rows = T * min(desc.top_k, Nd)
    if src.dtype != dst.dtype or src.shape[-1] != dst.shape[-1]:
        raise ValueError("src and dst must have the same dtype and row length")
    row_bytes = src.shape[-1] * src.element_size()
    i32 = torch.int32
    _call("occult_all_to_all", ctypes.byref(desc), int(n_src),
          _dev(counts, i32, n_src * Nd, "counts"), _dev(send_off, i32, n_src * Nd, "send_off"),
          _dev(recv_off, i32, n_src * Nd, "recv_off"),
          _dev(src, None, rows * src.shape[-1], "src"), _dev(dst, None, rows * dst.shape[-1], "dst"),
          ctypes.c_int64(row_bytes), int(bool(reverse)), _stream(stream))


def occult_profile_coact(desc, ids, n_tok, C, ws, P=None, vmask=None, ct_hist=None,
                         stream=None):
    Ne, k = desc.n_experts, desc.top_k
    max_ct = min(k, desc.n_vdev)
    need = workspace_size(desc, WS_PROFILE_COACT, n_tok)
    _call("occult_profile_coact", ctypes.byref(desc), _dev(ids, torch.int32, n_tok * k, "ids",
                                                            nullable=n_tok == 0),
          n_tok, _dev(vmask, torch.int32, n_tok, "vmask", nullable=True),
          _dev(C, torch.int64, Ne * Ne, "C"), _dev(P, torch.float32, Ne * Ne, "P", nullable=True),
          _dev(ct_hist, torch.int64, max_ct + 1, "ct_hist", nullable=True),
          _dev(ws, torch.uint8, need, "ws", nullable=need == 0), ctypes.c_size_t(need),
          _stream(stream))


from .pipeline import OccultMoE, desc_for  # noqa: E402  (needs the names above)
