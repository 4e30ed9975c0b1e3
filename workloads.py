"""Seeded synthetic workloads for routed-MoE expert execution.

This module only draws inputs: it holds none of the method's arithmetic, and
both the CUDA path's tests/bench and the CPU oracle take their inputs from it.

Workloads (T tokens, E experts, top-k, hidden H, intermediate I):

=========  =====  ===  ==  ====  ====  ==============================================
name         T     E   k    H     I    routing
=========  =====  ===  ==  ====  ====  ==============================================
tiny          64    8   2   256   512  k distinct uniform experts per token
decode1        1  384   6  7168  3072  k distinct uniform experts per token
decode8        8  384   6  7168  3072  k distinct uniform experts per token
small        128  256   8  7168  2048  k distinct, popularity p_e ~ (e+1)^-1.2 (Zipf)
prefill     2048  384   6  7168  3072  k distinct uniform experts per token
large       8192  128   8  4096  1536  25% of tokens: slot 0 = expert 0 and k-1
                                       distinct uniform from [1, E); the rest
                                       k distinct uniform from [0, E)
=========  =====  ===  ==  ====  ====  ==============================================

Values: x ~ N(0, 1), W13 and W2 ~ N(0, 0.02^2), drawn in fp32 by a seeded
``torch.Generator`` on the target device and rounded to bf16. Routing weights:
per-token logits ~ N(0, 1) over the k chosen experts, softmax over k (the
renormalised top-k softmax of a router), fp32. Routing is drawn on the host
with ``numpy.random.default_rng``. The shapes follow the expert counts, top-k,
hidden and intermediate sizes that the DeepGEMM MegaMoE page (Performance)
and the FlashInfer moe_ep page (benchmark tables) measure; nothing is read
from a dataset.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    E: int
    k: int
    H: int
    I: int
    routing: str          # "uniform" | "zipf" | "hot0"
    seed: int
    zipf_s: float = 1.2
    hot_frac: float = 0.25
    subset: int = 0       # tokens the oracle checks at full size (0 = all)

    @property
    def R(self) -> int:
        return self.T * self.k

    def describe(self) -> str:
        return (f"{self.name}: T={self.T} E={self.E} k={self.k} H={self.H} I={self.I} "
                f"routing={self.routing}")


WORKLOADS = {
    "tiny": Workload("tiny", 64, 8, 2, 256, 512, "uniform", seed=11),
    "decode1": Workload("decode1", 1, 384, 6, 7168, 3072, "uniform", seed=21),
    "decode8": Workload("decode8", 8, 384, 6, 7168, 3072, "uniform", seed=22),
    "small": Workload("small", 128, 256, 8, 7168, 2048, "zipf", seed=31),
    "prefill": Workload("prefill", 2048, 384, 6, 7168, 3072, "uniform", seed=41, subset=256),
    "large": Workload("large", 8192, 128, 8, 4096, 1536, "hot0", seed=51, subset=256),
}


def custom(name: str, T: int, E: int, k: int, H: int, I: int, routing: str = "uniform",
           seed: int = 0, **kw) -> Workload:
    return Workload(name, T, E, k, H, I, routing, seed=seed, **kw)


def _distinct_uniform(rng: np.random.Generator, n: int, E: int, k: int, low: int = 0) -> np.ndarray:
    """n rows of k distinct ids drawn uniformly from [low, E)."""
    if n == 0:
        return np.zeros((0, k), dtype=np.int32)
    keys = rng.random((n, E - low))
    return (np.argsort(keys, axis=1, kind="stable")[:, :k] + low).astype(np.int32)


def make_routing(wl: Workload, seed: int | None = None):
    """Return ``(topk_ids[T, k] int32, topk_weights[T, k] float32)`` as numpy arrays."""
    rng = np.random.default_rng(wl.seed if seed is None else seed)
    T, E, k = wl.T, wl.E, wl.k
    if wl.routing == "uniform":
        ids = _distinct_uniform(rng, T, E, k)
    elif wl.routing == "zipf":
        p = (np.arange(1, E + 1, dtype=np.float64)) ** (-wl.zipf_s)
        p /= p.sum()
        ids = np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
        ids = ids.reshape(T, k)
    elif wl.routing == "hot0":
        n_hot = int(round(T * wl.hot_frac))
        hot = np.zeros(T, dtype=bool)
        hot[rng.permutation(T)[:n_hot]] = True
        ids = np.empty((T, k), dtype=np.int32)
        ids[~hot] = _distinct_uniform(rng, int((~hot).sum()), E, k)
        ids[hot, 0] = 0
        ids[hot, 1:] = _distinct_uniform(rng, n_hot, E, k - 1, low=1)
    else:
        raise ValueError(f"unknown routing {wl.routing!r}")
    logits = rng.standard_normal((T, k))
    ex = np.exp(logits - logits.max(axis=1, keepdims=True)) if T else logits
    weights = (ex / ex.sum(axis=1, keepdims=True)).astype(np.float32) if T else logits.astype(np.float32)
    return np.ascontiguousarray(ids, dtype=np.int32), np.ascontiguousarray(weights, dtype=np.float32)


def _generator(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_x(wl: Workload, device="cpu", seed: int | None = None) -> torch.Tensor:
    """x[T, H] bf16 ~ N(0, 1)."""
    s = (wl.seed if seed is None else seed) * 7 + 1
    g = _generator(device, s)
    return torch.randn((wl.T, wl.H), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_weights(wl: Workload, device="cpu", seed: int | None = None, std: float = 0.02):
    """W13[E, 2I, H] and W2[E, H, I], bf16 ~ N(0, std^2), drawn expert by expert."""
    s = (wl.seed if seed is None else seed) * 7 + 2
    g = _generator(device, s)
    E, H, I = wl.E, wl.H, wl.I
    W13 = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device=device)
    W2 = torch.empty((E, H, I), dtype=torch.bfloat16, device=device)
    for e in range(E):
        W13[e] = torch.randn((2 * I, H), generator=g, device=device, dtype=torch.float32).mul_(std)
        W2[e] = torch.randn((H, I), generator=g, device=device, dtype=torch.float32).mul_(std)
    return W13, W2


def token_subset(wl: Workload, n: int | None = None) -> np.ndarray:
    """Seeded subset of tokens the oracle evaluates at full size (all tokens if none)."""
    n = wl.subset if n is None else n
    if not n or n >= wl.T:
        return np.arange(wl.T, dtype=np.int32)
    rng = np.random.default_rng(wl.seed + 1)
    return np.sort(rng.choice(wl.T, n, replace=False)).astype(np.int32)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """A bf16 tensor's bit patterns as a host uint16 array (no rounding)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
