"""CPU oracle for routed-MoE expert execution (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. The product path (the CUDA library and its
binding) never imports it, and this package imports nothing from the product.

The arithmetic lives in ``moe_oracle.c`` (plain loops, fp32, OpenMP across
independent rows); this module only marshals numpy arrays into it. What is
computed and which passage each step follows is written at the top of
``moe_oracle.c``:

* dispatch -- TileOps PR #1738 "Separate dispatched expert compute", Summary
  (local dispatch into a tight expert-major batch) and Scope (valid-row count
  read from ``expert_offsets[-1:]``);
* expert MLP -- same page, Summary (dispatched-expert MLP compute) and Review
  follow-up (fused-gated epilogue): ``a = bf16(SiLU(x W1^T) * (x W3^T))``,
  ``y = a W2^T`` in fp32;
* combine -- same page, Summary (routing weights kept outside expert compute):
  ``out = bf16(sum_j w_j y_j)`` in fp32, j ascending;
* MXFP8 weights -- FlashInfer moe_ep page (PR #3980), MXFP8 path with
  prequantized weights, format 32 e4m3 x e8m0 (OCP MX v1.0): ``mx_quantize``
  and the exact ``mx_dequantize``; the MXFP8 forward is the bf16 forward on
  dequantized weights.

Every function here is pinned by ``tests/test_oracle_pins.py`` against values
that do not come from the oracle itself (see that file's docstring).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import build_oracle, oracle_lib_path

__all__ = [
    "Oracle",
    "load",
    "round_bf16",
    "dispatch",
    "expert_rows",
    "combine_slots",
    "combine_sorted",
    "moe_tokens",
    "moe_forward_streamed",
    "bf16_bits_to_f32",
    "e4m3_values",
    "mx_quantize",
    "mx_dequantize",
]

_i32p = ctypes.POINTER(ctypes.c_int32)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray, ptype):
    return a.ctypes.data_as(ptype)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


class Oracle:
    """ctypes front of one build of ``moe_oracle.c``.

    The default instance (:func:`load`) wraps ``oracle/_build/liboracle.so``.
    Tests also wrap builds of deliberately mutated copies of the source to
    show that each pin catches a plausible mistake.
    """

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.oracle_round_bf16.argtypes = [ctypes.c_int64, _f32p, _u16p]
        lib.oracle_round_bf16.restype = None
        lib.oracle_dispatch.argtypes = [ctypes.c_int32, ctypes.c_int32, _i32p, _i32p, _i32p, _i32p, _i32p]
        lib.oracle_dispatch.restype = ctypes.c_int32
        lib.oracle_expert_rows.argtypes = [ctypes.c_int32, ctypes.c_int32, _u16p, _u16p, ctypes.c_int32,
                                           _u16p, _u16p, _f32p]
        lib.oracle_expert_rows.restype = None
        lib.oracle_combine_slots.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _f32p, _f32p,
                                             _i32p, _f32p, _u16p]
        lib.oracle_combine_slots.restype = None
        lib.oracle_combine_sorted.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _f32p, _i32p,
                                              _f32p, _f32p, _u16p]
        lib.oracle_combine_sorted.restype = None
        lib.oracle_moe_tokens.argtypes = [ctypes.c_int32] * 5 + [_u16p, _i32p, _f32p, _u16p, _u16p,
                                                                 ctypes.c_int32, _i32p, _f32p, _u16p]
        lib.oracle_moe_tokens.restype = ctypes.c_int32
        lib.oracle_e4m3_values.argtypes = [_f32p]
        lib.oracle_e4m3_values.restype = None
        lib.oracle_mx_quantize.argtypes = [ctypes.c_int64, ctypes.c_int32, _u16p, _u8p, _u8p]
        lib.oracle_mx_quantize.restype = None
        lib.oracle_mx_dequantize.argtypes = [ctypes.c_int64, ctypes.c_int32, _u8p, _u8p, _u16p]
        lib.oracle_mx_dequantize.restype = None
        self.lib = lib
        self.path = path

    def round_bf16(self, x: np.ndarray) -> np.ndarray:
        """float32 -> bf16 bit patterns, round to nearest, ties to even."""
        x = _c(x, np.float32)
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.oracle_round_bf16(x.size, _p(x, _f32p), _p(out, _u16p))
        return out

    def dispatch(self, topk_ids: np.ndarray, E: int):
        """Stable local dispatch of ``topk_ids[T, k]`` (int32).

        Returns ``(counts[E], offsets[E+1], perm[R], inv[R], n_bad)`` where
        ``perm[row] = slot`` for rows below ``offsets[E]`` (-1 after) and
        ``inv[slot] = row`` (-1 for a dropped slot).
        """
        ids = _c(topk_ids, np.int32).reshape(-1)
        R = ids.size
        counts = np.zeros(max(E, 1), dtype=np.int32)
        offsets = np.zeros(E + 1, dtype=np.int32)
        perm = np.full(max(R, 1), -1, dtype=np.int32)
        inv = np.full(max(R, 1), -1, dtype=np.int32)
        ids_buf = ids if R else np.zeros(1, np.int32)
        bad = self.lib.oracle_dispatch(R, E, _p(ids_buf, _i32p), _p(counts, _i32p), _p(offsets, _i32p),
                                       _p(perm, _i32p), _p(inv, _i32p))
        return counts[:E], offsets, perm[:R], inv[:R], int(bad)

    def expert_rows(self, x_rows: np.ndarray, W13e: np.ndarray, W2e: np.ndarray):
        """Rows ``x_rows[n, H]`` (bf16 bits) through one expert.

        ``W13e[2I, H]`` and ``W2e[H, I]`` are bf16 bits. Returns ``(a[n, I] bf16
        bits, y[n, H] float32)``.
        """
        x_rows = _c(x_rows, np.uint16)
        W13e = _c(W13e, np.uint16)
        W2e = _c(W2e, np.uint16)
        n, H = x_rows.shape
        I = W13e.shape[0] // 2
        assert W13e.shape == (2 * I, H) and W2e.shape == (H, I)
        a = np.empty((n, I), dtype=np.uint16)
        y = np.empty((n, H), dtype=np.float32)
        if n:
            self.lib.oracle_expert_rows(H, I, _p(W13e, _u16p), _p(W2e, _u16p), n, _p(x_rows, _u16p),
                                        _p(a, _u16p), _p(y, _f32p))
        return a, y

    def combine_slots(self, y_slot: np.ndarray, w: np.ndarray, valid: np.ndarray):
        """``y_slot[n, k, H]`` fp32, ``w[n, k]``, ``valid[n, k]`` -> (out_acc fp32, out bf16 bits)."""
        y_slot = _c(y_slot, np.float32)
        w = _c(w, np.float32)
        valid = _c(valid, np.int32)
        n, k, H = y_slot.shape
        out_acc = np.empty((n, H), dtype=np.float32)
        out = np.empty((n, H), dtype=np.uint16)
        if n:
            self.lib.oracle_combine_slots(n, k, H, _p(y_slot, _f32p), _p(w, _f32p), _p(valid, _i32p),
                                          _p(out_acc, _f32p), _p(out, _u16p))
        return out_acc, out

    def combine_sorted(self, y_sorted: np.ndarray, inv: np.ndarray, w: np.ndarray):
        """Combine from the expert-major batch ``y_sorted[rows, H]`` (fp32) via ``inv[T*k]``."""
        y_sorted = _c(y_sorted, np.float32)
        w = _c(w, np.float32)
        T, k = w.shape
        H = y_sorted.shape[1]
        inv = _c(inv, np.int32).reshape(-1)
        assert inv.size == T * k
        out_acc = np.empty((T, H), dtype=np.float32)
        out = np.empty((T, H), dtype=np.uint16)
        if T:
            self.lib.oracle_combine_sorted(T, k, H, _p(y_sorted, _f32p), _p(inv, _i32p), _p(w, _f32p),
                                           _p(out_acc, _f32p), _p(out, _u16p))
        return out_acc, out

    def moe_tokens(self, x, topk_ids, topk_weights, W13, W2, tokens=None):
        """Whole forward for the listed tokens, all inputs host-resident.

        ``x[T, H]``, ``W13[E, 2I, H]``, ``W2[E, H, I]`` are bf16 bits (uint16);
        ``topk_ids[T, k]`` int32, ``topk_weights[T, k]`` float32. Returns
        ``(out_acc[n, H] fp32, out[n, H] bf16 bits, n_bad_ids)``.
        """
        x = _c(x, np.uint16)
        ids = _c(topk_ids, np.int32)
        w = _c(topk_weights, np.float32)
        W13 = _c(W13, np.uint16)
        W2 = _c(W2, np.uint16)
        T, H = x.shape
        E, twoI, _ = W13.shape
        I = twoI // 2
        k = ids.shape[1]
        tok = np.arange(T, dtype=np.int32) if tokens is None else _c(tokens, np.int32)
        n = tok.size
        out_acc = np.empty((n, H), dtype=np.float32)
        out = np.empty((n, H), dtype=np.uint16)
        bad = 0
        if n:
            bad = self.lib.oracle_moe_tokens(T, E, k, H, I, _p(x, _u16p), _p(ids, _i32p), _p(w, _f32p),
                                             _p(W13, _u16p), _p(W2, _u16p), n, _p(tok, _i32p),
                                             _p(out_acc, _f32p), _p(out, _u16p))
        return out_acc, out, int(bad)

    def e4m3_values(self) -> np.ndarray:
        """float32[256]: the value of every E4M3 code (NaN for 0x7F and 0xFF)."""
        out = np.empty(256, dtype=np.float32)
        self.lib.oracle_e4m3_values(_p(out, _f32p))
        return out

    def mx_quantize(self, w: np.ndarray):
        """MXFP8 quantization along the last axis of bf16 bits ``w[..., K]``
        (K a multiple of 32): returns ``(q[..., K] E4M3 codes, s[..., K/32]
        E8M0 scale codes)``, both uint8."""
        w = _c(w, np.uint16)
        K = w.shape[-1]
        assert K % 32 == 0
        rows = w.size // K
        q = np.empty(w.shape, dtype=np.uint8)
        s = np.empty(w.shape[:-1] + (K // 32,), dtype=np.uint8)
        if rows:
            self.lib.oracle_mx_quantize(rows, K, _p(w, _u16p), _p(q, _u8p), _p(s, _u8p))
        return q, s

    def mx_dequantize(self, q: np.ndarray, s: np.ndarray) -> np.ndarray:
        """bf16 bits of X * P for MXFP8 codes ``q[..., K]`` and scales ``s[..., K/32]``."""
        q = _c(q, np.uint8)
        s = _c(s, np.uint8)
        K = q.shape[-1]
        assert s.shape == q.shape[:-1] + (K // 32,)
        rows = q.size // K
        out = np.empty(q.shape, dtype=np.uint16)
        if rows:
            self.lib.oracle_mx_dequantize(rows, K, _p(q, _u8p), _p(s, _u8p), _p(out, _u16p))
        return out

    def moe_forward_streamed(self, x, topk_ids, topk_weights, fetch_expert, E, tokens=None):
        """Same result as :meth:`moe_tokens`, with expert weights fetched one at a time.

        For workloads whose weights do not fit comfortably in host memory:
        ``fetch_expert(e)`` returns ``(W13e[2I, H], W2e[H, I])`` as bf16 bits.
        Each expert's rows go through :meth:`expert_rows` (the same per-row C
        routine as :meth:`moe_tokens`), then :meth:`combine_slots` sums the k
        slots of each token in ascending j, so the two agree bit for bit.
        """
        x = _c(x, np.uint16)
        ids = _c(topk_ids, np.int32)
        w = _c(topk_weights, np.float32)
        T, H = x.shape
        k = ids.shape[1]
        tok = np.arange(T, dtype=np.int32) if tokens is None else _c(tokens, np.int32)
        n = tok.size
        sub_ids = ids[tok]
        valid = ((sub_ids >= 0) & (sub_ids < E)).astype(np.int32)
        y_slot = np.zeros((n, k, H), dtype=np.float32)
        for e in np.unique(sub_ids[valid.astype(bool)]):
            qs, js = np.nonzero(sub_ids == e)
            W13e, W2e = fetch_expert(int(e))
            _, y = self.expert_rows(x[tok[qs]], W13e, W2e)
            y_slot[qs, js] = y
        return self.combine_slots(y_slot, w[tok], valid)


_default = None


def load() -> Oracle:
    """Build (if needed) and load the default oracle library."""
    global _default
    if _default is None:
        path = oracle_lib_path()
        if not os.path.exists(path):
            build_oracle()
        _default = Oracle(path)
    return _default


def round_bf16(x):
    return load().round_bf16(x)


def dispatch(topk_ids, E):
    return load().dispatch(topk_ids, E)


def expert_rows(x_rows, W13e, W2e):
    return load().expert_rows(x_rows, W13e, W2e)


def combine_slots(y_slot, w, valid):
    return load().combine_slots(y_slot, w, valid)


def combine_sorted(y_sorted, inv, w):
    return load().combine_sorted(y_sorted, inv, w)


def moe_tokens(x, topk_ids, topk_weights, W13, W2, tokens=None):
    return load().moe_tokens(x, topk_ids, topk_weights, W13, W2, tokens)


def moe_forward_streamed(x, topk_ids, topk_weights, fetch_expert, E, tokens=None):
    return load().moe_forward_streamed(x, topk_ids, topk_weights, fetch_expert, E, tokens)


def e4m3_values():
    return load().e4m3_values()


def mx_quantize(w):
    return load().mx_quantize(w)


def mx_dequantize(q, s):
    return load().mx_dequantize(q, s)
