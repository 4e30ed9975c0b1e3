"""GPU parity of the two tcgen05 grouped GEMMs (moe_expert_compute) against the
oracle's per-expert MLP, on both paths and every token-tile height, with
several tiles and ragged expert segments."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as wlm
from parity import assert_within_tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from moe_routed_expert_routing_gb300.build import build
    build()
    from moe_routed_expert_routing_gb300 import binding
    return binding


def dispatch_and_compute(B, p, ids_np, x, W13, W2):
    offs = torch.empty(p.E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(p.cap, dtype=torch.int32, device="cuda")
    inv = torch.empty(p.T_max * p.k, dtype=torch.int32, device="cuda")
    ws = torch.zeros(B.moe_workspace_size(p), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((p.cap, p.H), dtype=torch.bfloat16, device="cuda")
    ys = torch.full((p.cap, p.H), float("nan"), dtype=torch.float32, device="cuda")
    B.moe_dispatch(p, torch.from_numpy(ids_np).cuda(), offs, perm, inv, ws, x=x, x_sorted=xs)
    B.moe_expert_compute(p, xs, offs, W13, W2, ys, ws)
    torch.cuda.synchronize()
    assert B.moe_last_device_error(ws) == 0
    return offs.cpu().numpy(), xs, ys


def oracle_y(offs, xs, W13, W2, E):
    """The oracle's fp32 y for every valid row of the sorted batch."""
    n = int(offs[-1])
    y = np.zeros((n, xs.shape[1]), dtype=np.float32)
    xs_np = wlm.bf16_bits(xs[:n])
    for e in range(E):
        a, b = int(offs[e]), int(offs[e + 1])
        if b > a:
            _, y[a:b] = oracle.expert_rows(xs_np[a:b], wlm.bf16_bits(W13[e]), wlm.bf16_bits(W2[e]))
    return y


CASES = [
    # name, T, E, k, H, I, path, routing
    ("tiled_small", 96, 4, 2, 256, 256, 1, "uniform"),          # 48 rows/expert: ragged 128-row tiles
    ("tiled_multi", 300, 3, 2, 512, 384, 1, "uniform"),         # 200 rows/expert: 2 tiles each
    ("tiled_skew", 400, 8, 2, 256, 512, 1, "hot0"),             # one hot expert, several m-tiles
    ("small16", 8, 64, 4, 512, 256, 2, "uniform"),             # token tile 16
    ("small32", 40, 32, 4, 256, 384, 2, "uniform"),            # token tile 32
    ("small64", 120, 16, 4, 256, 256, 2, "uniform"),           # token tile 64, rows > 64 per expert
    ("small_zipf", 128, 64, 8, 512, 256, 2, "zipf"),           # empty experts + heavy ones
    ("tiny_tiled", 64, 8, 2, 256, 512, 1, "uniform"),
    ("tiny_small", 64, 8, 2, 256, 512, 2, "uniform"),
    ("tiled1_small", 96, 4, 2, 256, 256, 3, "uniform"),         # single-CTA tiles
    ("tiled1_skew", 400, 8, 2, 256, 512, 3, "hot0"),
    ("pair_multi", 700, 3, 2, 512, 384, 1, "uniform"),          # ~467 rows/expert: 2 pair tiles, ragged
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_expert_compute_matches_oracle(B, case):
    name, T, E, k, H, I, path, routing = case
    wl = wlm.custom(name, T, E, k, H, I, routing=routing, seed=T * 7 + E)
    ids_np, _ = wlm.make_routing(wl)
    x = wlm.make_x(wl, "cuda")
    W13, W2 = wlm.make_weights(wl, "cuda")
    p = B.Problem.make(T, E, k, H, I, path=path)
    offs, xs, ys = dispatch_and_compute(B, p, ids_np, x, W13, W2)
    ref = oracle_y(offs, xs, W13, W2, E)
    n = int(offs[-1])
    assert_within_tolerance(ys[:n].cpu().numpy(), ref, name)


@pytest.mark.parametrize("path", [1, 2, 3])
def test_gate_up_stage_alone(B, path):
    """W2 = identity (H == I): y equals the activation h, so the gate-up GEMM and
    its SiLU(gate)*up epilogue are checked on their own, nearly bit for bit."""
    T, E, k, H, I = 160, 4, 2, 256, 256
    wl = wlm.custom("gu", T, E, k, H, I, seed=77)
    ids_np, _ = wlm.make_routing(wl)
    x = wlm.make_x(wl, "cuda")
    W13, _ = wlm.make_weights(wl, "cuda", std=0.05)
    W2 = torch.eye(H, dtype=torch.bfloat16, device="cuda").expand(E, H, I).contiguous()
    p = B.Problem.make(T, E, k, H, I, path=path)
    offs, xs, ys = dispatch_and_compute(B, p, ids_np, x, W13, W2)
    n = int(offs[-1])
    xs_np = wlm.bf16_bits(xs[:n])
    a_ref = np.zeros((n, I), dtype=np.uint16)
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi > lo:
            a_ref[lo:hi], _ = oracle.expert_rows(xs_np[lo:hi], wlm.bf16_bits(W13[e]), wlm.bf16_bits(W2[e]))
    got = ys[:n].double().cpu().numpy()
    ref = oracle.bf16_bits_to_f32(a_ref).astype(np.float64)
    # Both sides round SiLU(g)*u to bf16 from fp32 sums taken in different
    # orders. Allowed difference: one bf16 ulp of the reference plus the
    # forward-error bound of the two fp32 sums of H terms, propagated through
    # SiLU(g)*u (large only where the sums cancel).
    eps = 2.0 ** -24
    xsf = xs[:n].double().abs()
    dg = torch.zeros((n, I), dtype=torch.float64, device="cuda")
    du = torch.zeros_like(dg)
    gu = torch.zeros_like(dg)
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi > lo:
            W1 = W13[e, :I].double()
            W3 = W13[e, I:].double()
            dg[lo:hi] = H * eps * (xsf[lo:hi] @ W1.abs().T)
            du[lo:hi] = H * eps * (xsf[lo:hi] @ W3.abs().T) * torch.nn.functional.silu(xs[lo:hi].double() @ W1.T).abs()
            gu[lo:hi] = (xs[lo:hi].double() @ W3.T).abs()
    bound = (1.1 * dg * gu + du).cpu().numpy()
    ulp = 2.0 * np.abs(ref) * 2.0 ** -8 + 1e-30
    diff = np.abs(got - ref)
    assert np.all(diff <= ulp + bound), float((diff - ulp - bound).max())
    assert np.count_nonzero(diff) <= max(4, diff.size // 200), np.count_nonzero(diff)
