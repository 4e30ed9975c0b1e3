"""Shared helpers for the parity tests: run a workload through the CUDA path
and through the oracle, and compare with the stated tolerance.

Tolerance for the MoE output (routed-MoE problem statement): over the
compared elements,
  * max |out - ref| <= 1e-2 * rms(ref) + 1e-3, where ref is the oracle's fp32
    accumulator and the GPU output's own final rounding to bf16 (half an ulp
    of bf16 at ref, at most 2^-9 |ref|) is allowed on top -- no bf16 output
    could meet the bound without it;
  * mean relative error sum|out - ref| / sum|ref| <= 5e-3.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as wlm

MAX_ERR_REL_RMS = 1e-2
MAX_ERR_ABS = 1e-3
MEAN_REL_ERR = 5e-3


def bf16_half_ulp(ref: np.ndarray) -> np.ndarray:
    """Half an ulp of bf16 at |ref| (8 significant bits)."""
    a = np.abs(ref.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 1e-38)))
    return np.where(a > 0, 2.0 ** (e - 8), 0.0)


def error_metrics(got_bf16_bits: np.ndarray, ref_f32: np.ndarray) -> dict:
    """Error of a bf16 result (bit patterns, uint16) or an fp32 result against ref."""
    if got_bf16_bits.dtype == np.uint16:
        got = oracle.bf16_bits_to_f32(got_bf16_bits).astype(np.float64)
    else:
        got = np.asarray(got_bf16_bits, dtype=np.float64)
    ref = ref_f32.astype(np.float64)
    err = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    excess = err - bf16_half_ulp(ref) if got_bf16_bits.dtype == np.uint16 else err
    return {
        "max_err": float(err.max()) if err.size else 0.0,
        "max_err_beyond_output_rounding": float(excess.max()) if err.size else 0.0,
        "bound": MAX_ERR_REL_RMS * rms + MAX_ERR_ABS,
        "rms_ref": rms,
        "mean_rel_err": float(err.sum() / max(np.abs(ref).sum(), 1e-30)),
        "rel_l2": float(np.sqrt((err ** 2).sum() / max((ref ** 2).sum(), 1e-30))),
        "n": int(err.size),
        "finite": bool(np.all(np.isfinite(got))),
    }


def assert_within_tolerance(got_bf16_bits, ref_f32, what=""):
    m = error_metrics(got_bf16_bits, ref_f32)
    assert m["finite"], f"{what}: non-finite output {m}"
    assert m["max_err_beyond_output_rounding"] <= m["bound"], f"{what}: max error {m}"
    assert m["mean_rel_err"] <= MEAN_REL_ERR, f"{what}: mean relative error {m}"
    return m


class DeviceWorkload:
    """A workload's inputs resident on the GPU plus host copies of routing."""

    def __init__(self, wl: wlm.Workload, device="cuda", seed=None):
        self.wl = wl
        self.device = device
        self.ids_np, self.w_np = wlm.make_routing(wl, seed)
        self.x = wlm.make_x(wl, device, seed)
        self.W13, self.W2 = wlm.make_weights(wl, device, seed)
        self.ids = torch.from_numpy(self.ids_np).to(device)
        self.w = torch.from_numpy(self.w_np).to(device)

    def fetch_expert(self, e: int):
        return wlm.bf16_bits(self.W13[e]), wlm.bf16_bits(self.W2[e])

    def oracle_out(self, tokens=None, ids_np=None, w_np=None):
        """Oracle (out_acc fp32, out bf16 bits) for the listed tokens."""
        ids_np = self.ids_np if ids_np is None else ids_np
        w_np = self.w_np if w_np is None else w_np
        x = wlm.bf16_bits(self.x)
        return oracle.moe_forward_streamed(x, ids_np, w_np, self.fetch_expert, self.wl.E, tokens)
