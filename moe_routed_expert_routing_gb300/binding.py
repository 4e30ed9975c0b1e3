"""Thin ctypes binding of libmoe.so (the C ABI in include/moe.h).

Argument marshalling only: every step of routed expert execution runs in the
library's CUDA kernels. Torch tensors supply device memory and the current
stream; their pointers go straight to the C entry points, which keep the same
names here. If libmoe.so is missing this module raises at load time -- there
is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import lib_path

MOE_OK = 0
MOE_PATH_AUTO = 0
MOE_PATH_TILED = 1
MOE_PATH_SMALL_M = 2
MOE_PATH_TILED_1CTA = 3
MOE_WEIGHTS_ROW_MAJOR = 0
MOE_WEIGHTS_PACKED = 1
MOE_WEIGHTS_MXFP8 = 2
MOE_FORWARD_AUTO = 0
MOE_FORWARD_SEPARATE = 1
MOE_FORWARD_ONE_KERNEL = 2
MOE_DEVERR_BAD_EXPERT_ID = 0x1
MOE_DEVERR_WAIT_TIMEOUT = 0x2
MOE_DEVERR_Y_RANGE = 0x4

#: every symbol include/moe.h declares
EXPORTED_SYMBOLS = (
    "moe_workspace_size",
    "moe_resolve_path",
    "moe_resolve_profile",
    "moe_dispatch",
    "moe_expert_compute",
    "moe_combine",
    "moe_forward",
    "moe_forward_profiled",
    "moe_dispatch_noalloc",
    "moe_pack_weights",
    "moe_weight_bytes",
    "moe_quantize_weights",
    "moe_last_device_error",
    "moe_clear_device_error",
    "moe_status_string",
)


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


class Problem(ctypes.Structure):
    """``moe_problem_t``: T_max, E, k, H, I, capacity (0 = T_max*k), path."""

    _fields_ = [
        ("T_max", ctypes.c_int32),
        ("E", ctypes.c_int32),
        ("k", ctypes.c_int32),
        ("H", ctypes.c_int32),
        ("I", ctypes.c_int32),
        ("capacity", ctypes.c_int32),
        ("path", ctypes.c_int32),
        ("weight_layout", ctypes.c_int32),
        ("forward_form", ctypes.c_int32),
    ]

    @classmethod
    def make(cls, T_max, E, k, H, I, capacity=0, path=MOE_PATH_AUTO, weight_layout=MOE_WEIGHTS_ROW_MAJOR,
             forward_form=MOE_FORWARD_AUTO):
        return cls(int(T_max), int(E), int(k), int(H), int(I), int(capacity), int(path), int(weight_layout),
                   int(forward_form))

    @property
    def cap(self) -> int:
        return self.capacity or self.T_max * self.k

    def __repr__(self):
        return (f"Problem(T_max={self.T_max}, E={self.E}, k={self.k}, H={self.H}, I={self.I}, "
                f"capacity={self.capacity}, path={self.path}, weight_layout={self.weight_layout}, "
                f"forward_form={self.forward_form})")


class Profile(ctypes.Structure):
    """``moe_profile_t``: the static launch profile of a problem."""

    _fields_ = [("path", ctypes.c_int32), ("tile_rows", ctypes.c_int32), ("down_split_k", ctypes.c_int32),
                ("pdl", ctypes.c_int32), ("fused_gather", ctypes.c_int32), ("cta_pair", ctypes.c_int32),
                ("fused_mlp", ctypes.c_int32), ("megakernel", ctypes.c_int32),
                ("kernel_launches", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {n: getattr(self, n) for n, _ in self._fields_}


_lib = None
_vp = ctypes.c_void_p
_P = ctypes.POINTER(Problem)


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libmoe.so (built by ``build.build()``); raise if it is absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or lib_path()
    if not os.path.exists(p):
        raise RuntimeError(f"libmoe.so not found at {p}: run moe_routed_expert_routing_gb300.build.build() "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(p)
    st = ctypes.c_int
    lib.moe_workspace_size.argtypes = [_P, ctypes.POINTER(ctypes.c_size_t)]
    lib.moe_workspace_size.restype = st
    lib.moe_resolve_path.argtypes = [_P, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
    lib.moe_resolve_path.restype = st
    lib.moe_resolve_profile.argtypes = [_P, ctypes.POINTER(Profile)]
    lib.moe_resolve_profile.restype = st
    lib.moe_dispatch.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.moe_dispatch.restype = st
    lib.moe_expert_compute.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.moe_expert_compute.restype = st
    lib.moe_combine.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.moe_combine.restype = st
    lib.moe_forward.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.moe_forward.restype = st
    lib.moe_forward_profiled.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t,
                                         _vp, ctypes.POINTER(_vp)]
    lib.moe_forward_profiled.restype = st
    lib.moe_dispatch_noalloc.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.moe_dispatch_noalloc.restype = st
    lib.moe_pack_weights.argtypes = [_P, _vp, _vp, _vp, _vp, _vp]
    lib.moe_pack_weights.restype = st
    lib.moe_weight_bytes.argtypes = [_P, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t),
                                     ctypes.POINTER(ctypes.c_size_t)]
    lib.moe_weight_bytes.restype = st
    lib.moe_quantize_weights.argtypes = [_P, _vp, _vp, _vp, _vp, _vp]
    lib.moe_quantize_weights.restype = st
    lib.moe_last_device_error.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_int32)]
    lib.moe_last_device_error.restype = st
    lib.moe_clear_device_error.argtypes = [_vp, _vp]
    lib.moe_clear_device_error.restype = st
    lib.moe_status_string.argtypes = [ctypes.c_int]
    lib.moe_status_string.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load_library().moe_status_string(int(status)).decode()
    except Exception:  # pragma: no cover - library absent
        return f"status {status}"


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors passed to libmoe must be contiguous")
    return t.data_ptr()


def _need(t, name: str, dtype, numel: int):
    """Fail closed before any launch: ``t`` must be a CUDA tensor of ``dtype``
    with at least ``numel`` elements. The C entry points see plain pointers
    and cannot check the extent of a buffer; a short one would be read or
    written out of bounds on the device. (A raw int pointer is passed on
    unchecked, as the C caller's responsibility.)"""
    if t is None or isinstance(t, int):
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (device memory), not on {t.device}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, not {t.dtype}")
    if t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements; the problem needs at least {numel}")


def _need_weights(problem, W13, W2):
    """W13 [E, 2I, H] and W2 [E, H, I] in the problem's weight layout."""
    if problem.weight_layout == MOE_WEIGHTS_MXFP8:
        b13, b2 = moe_weight_bytes(problem, MOE_WEIGHTS_MXFP8)
        _need(W13, "W13", torch.uint8, b13)
        _need(W2, "W2", torch.uint8, b2)
    else:
        _need(W13, "W13", torch.bfloat16, problem.E * 2 * problem.I * problem.H)
        _need(W2, "W2", torch.bfloat16, problem.E * problem.H * problem.I)


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(status, what)


def moe_workspace_size(problem: Problem) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().moe_workspace_size(ctypes.byref(problem), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def moe_resolve_path(problem: Problem):
    path = ctypes.c_int32(0)
    rows = ctypes.c_int32(0)
    _check(load_library().moe_resolve_path(ctypes.byref(problem), ctypes.byref(path), ctypes.byref(rows)),
           "moe_resolve_path")
    return path.value, rows.value


def moe_resolve_profile(problem: Problem) -> dict:
    prof = Profile()
    _check(load_library().moe_resolve_profile(ctypes.byref(problem), ctypes.byref(prof)), "moe_resolve_profile")
    return prof.as_dict()


def _need_routing(problem, topk_ids, expert_offsets, perm, d_num_tokens):
    R = problem.T_max * problem.k
    _need(topk_ids, "topk_ids", torch.int32, R)
    _need(expert_offsets, "expert_offsets", torch.int32, problem.E + 1)
    _need(perm, "perm", torch.int32, problem.cap)
    _need(d_num_tokens, "d_num_tokens", torch.int32, 1)


def moe_dispatch(problem, topk_ids, expert_offsets, perm, inv, ws, x=None, x_sorted=None, d_num_tokens=None,
                 stream=None):
    _need_routing(problem, topk_ids, expert_offsets, perm, d_num_tokens)
    _need(inv, "inv", torch.int32, problem.T_max * problem.k)
    _need(ws, "ws", None, 0)
    _need(x, "x", torch.bfloat16, problem.T_max * problem.H)
    _need(x_sorted, "x_sorted", torch.bfloat16, problem.cap * problem.H)
    _check(load_library().moe_dispatch(ctypes.byref(problem), _ptr(topk_ids), _ptr(d_num_tokens),
                                       _ptr(expert_offsets), _ptr(perm), _ptr(inv), _ptr(x), _ptr(x_sorted),
                                       _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "moe_dispatch")


def moe_dispatch_noalloc(problem, topk_ids, expert_offsets, perm, inv, x=None, x_sorted=None, d_num_tokens=None,
                         stream=None):
    """moe_dispatch with no workspace (library-owned static scratch); see include/moe.h."""
    _need_routing(problem, topk_ids, expert_offsets, perm, d_num_tokens)
    _need(inv, "inv", torch.int32, problem.T_max * problem.k)
    _need(x, "x", torch.bfloat16, problem.T_max * problem.H)
    _need(x_sorted, "x_sorted", torch.bfloat16, problem.cap * problem.H)
    _check(load_library().moe_dispatch_noalloc(ctypes.byref(problem), _ptr(topk_ids), _ptr(d_num_tokens),
                                               _ptr(expert_offsets), _ptr(perm), _ptr(inv), _ptr(x),
                                               _ptr(x_sorted), _stream(stream)), "moe_dispatch_noalloc")


def moe_expert_compute(problem, x_sorted, expert_offsets, W13, W2, y_sorted, ws, stream=None):
    _need(x_sorted, "x_sorted", torch.bfloat16, problem.cap * problem.H)
    _need(expert_offsets, "expert_offsets", torch.int32, problem.E + 1)
    if problem.weight_layout != MOE_WEIGHTS_MXFP8:   # that layout is refused by the library itself
        _need_weights(problem, W13, W2)
    _need(y_sorted, "y_sorted", torch.float32, problem.cap * problem.H)
    _need(ws, "ws", None, 0)
    _check(load_library().moe_expert_compute(ctypes.byref(problem), _ptr(x_sorted), _ptr(expert_offsets), _ptr(W13),
                                             _ptr(W2), _ptr(y_sorted), _ptr(ws), ws.numel() * ws.element_size(),
                                             _stream(stream)), "moe_expert_compute")


def moe_combine(problem, y_sorted, inv, topk_weights, out, d_num_tokens=None, stream=None):
    _need(y_sorted, "y_sorted", torch.float32, problem.cap * problem.H)
    _need(inv, "inv", torch.int32, problem.T_max * problem.k)
    _need(topk_weights, "topk_weights", torch.float32, problem.T_max * problem.k)
    _need(out, "out", torch.bfloat16, problem.T_max * problem.H)
    _need(d_num_tokens, "d_num_tokens", torch.int32, 1)
    _check(load_library().moe_combine(ctypes.byref(problem), _ptr(y_sorted), _ptr(inv), _ptr(topk_weights),
                                      _ptr(d_num_tokens), _ptr(out), _stream(stream)), "moe_combine")


def _need_forward(problem, x, topk_ids, topk_weights, W13, W2, expert_offsets, perm, out, ws, d_num_tokens):
    _need(x, "x", torch.bfloat16, problem.T_max * problem.H)
    _need_routing(problem, topk_ids, expert_offsets, perm, d_num_tokens)
    _need(topk_weights, "topk_weights", torch.float32, problem.T_max * problem.k)
    _need_weights(problem, W13, W2)
    _need(out, "out", torch.bfloat16, problem.T_max * problem.H)
    _need(ws, "ws", None, 0)


def moe_forward(problem, x, topk_ids, topk_weights, W13, W2, expert_offsets, perm, out, ws, d_num_tokens=None,
                stream=None):
    _need_forward(problem, x, topk_ids, topk_weights, W13, W2, expert_offsets, perm, out, ws, d_num_tokens)
    _check(load_library().moe_forward(ctypes.byref(problem), _ptr(x), _ptr(topk_ids), _ptr(topk_weights),
                                      _ptr(d_num_tokens), _ptr(W13), _ptr(W2), _ptr(expert_offsets), _ptr(perm),
                                      _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_forward")


def moe_forward_profiled(problem, x, topk_ids, topk_weights, W13, W2, expert_offsets, perm, out, ws, events,
                         d_num_tokens=None, stream=None):
    """moe_forward plus 6 stage events (torch.cuda.Event(enable_timing=True), already recorded once)."""
    _need_forward(problem, x, topk_ids, topk_weights, W13, W2, expert_offsets, perm, out, ws, d_num_tokens)
    arr = (_vp * 6)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(load_library().moe_forward_profiled(ctypes.byref(problem), _ptr(x), _ptr(topk_ids), _ptr(topk_weights),
                                               _ptr(d_num_tokens), _ptr(W13), _ptr(W2), _ptr(expert_offsets),
                                               _ptr(perm), _ptr(out), _ptr(ws), ws.numel() * ws.element_size(),
                                               _stream(stream), arr), "moe_forward_profiled")


def moe_pack_weights(problem, W13, W2, W13_packed=None, W2_packed=None, stream=None):
    """Reorder W13/W2 into the PACKED layout; returns (W13_packed, W2_packed)."""
    if W13_packed is None:
        W13_packed = torch.empty_like(W13)
    if W2_packed is None:
        W2_packed = torch.empty_like(W2)
    for name, t in (("W13", W13), ("W2", W2), ("W13_packed", W13_packed), ("W2_packed", W2_packed)):
        _need(t, name, torch.bfloat16, problem.E * (2 if "13" in name else 1) * problem.I * problem.H)
    _check(load_library().moe_pack_weights(ctypes.byref(problem), _ptr(W13), _ptr(W2), _ptr(W13_packed),
                                           _ptr(W2_packed), _stream(stream)), "moe_pack_weights")
    return W13_packed, W2_packed


def moe_weight_bytes(problem, layout):
    """(W13 bytes, W2 bytes) of the weights in ``layout``."""
    a, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(load_library().moe_weight_bytes(ctypes.byref(problem), int(layout), ctypes.byref(a), ctypes.byref(b)),
           "moe_weight_bytes")
    return a.value, b.value


def moe_quantize_weights(problem, W13, W2, W13_mx=None, W2_mx=None, stream=None):
    """Quantize row-major bf16 W13/W2 to the MXFP8 layout; returns (W13_mx, W2_mx) uint8 buffers."""
    b13, b2 = moe_weight_bytes(problem, MOE_WEIGHTS_MXFP8)
    if W13_mx is None:
        W13_mx = torch.empty(b13, dtype=torch.uint8, device=W13.device)
    if W2_mx is None:
        W2_mx = torch.empty(b2, dtype=torch.uint8, device=W2.device)
    _need(W13, "W13", torch.bfloat16, problem.E * 2 * problem.I * problem.H)
    _need(W2, "W2", torch.bfloat16, problem.E * problem.H * problem.I)
    _need(W13_mx, "W13_mx", torch.uint8, b13)
    _need(W2_mx, "W2_mx", torch.uint8, b2)
    _check(load_library().moe_quantize_weights(ctypes.byref(problem), _ptr(W13), _ptr(W2), _ptr(W13_mx),
                                               _ptr(W2_mx), _stream(stream)), "moe_quantize_weights")
    return W13_mx, W2_mx


def moe_last_device_error(ws, stream=None) -> int:
    _need(ws, "ws", None, 4)
    code = ctypes.c_int32(0)
    _check(load_library().moe_last_device_error(_ptr(ws), _stream(stream), ctypes.byref(code)),
           "moe_last_device_error")
    return code.value


def moe_clear_device_error(ws, stream=None):
    _need(ws, "ws", None, 0)
    _check(load_library().moe_clear_device_error(_ptr(ws), _stream(stream)), "moe_clear_device_error")


class Buffers:
    """Caller-owned device buffers for one problem (plumbing for tests and bench)."""

    def __init__(self, problem: Problem, device="cuda"):
        p = problem
        dev = torch.device(device)
        self.problem = p
        self.ws = torch.empty(moe_workspace_size(p), dtype=torch.uint8, device=dev)
        self.expert_offsets = torch.empty(p.E + 1, dtype=torch.int32, device=dev)
        self.perm = torch.empty(p.cap, dtype=torch.int32, device=dev)
        self.inv = torch.empty(p.T_max * p.k, dtype=torch.int32, device=dev)
        self.x_sorted = torch.empty((p.cap, p.H), dtype=torch.bfloat16, device=dev)
        self.y_sorted = torch.empty((p.cap, p.H), dtype=torch.float32, device=dev)
        self.out = torch.empty((p.T_max, p.H), dtype=torch.bfloat16, device=dev)
        self.ws.zero_()
