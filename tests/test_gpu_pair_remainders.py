"""The CTA-pair GEMMs on every kind of last row tile: an expert's last tile of
at most 128 rows runs swapped (weights on the MMA's M side, its rows on N),
longer ones run as 256-row tiles. Expert row counts are chosen around those
edges (1, 15/16/17, 31/32/33, 63/64/65, 127/128/129, 200, 239/240/241,
255/256/257, several tiles ending in 129, 193 or 255 rows, none), and the
outputs of both GEMMs and of the whole forward are checked against the
oracle, with H and I multiples of 64 that are not multiples of 128."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as wlm
from parity import assert_within_tolerance

pytestmark = pytest.mark.gpu

COUNTS = [1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 200, 239, 240, 241, 255, 256, 257, 0, 385, 449,
          511, 640]


@pytest.fixture(scope="module")
def B():
    from moe_routed_expert_routing_gb300.build import build
    build()
    from moe_routed_expert_routing_gb300 import binding
    return binding


def routing(counts, seed):
    """k = 1: expert e gets counts[e] tokens, in a shuffled token order."""
    ids = np.repeat(np.arange(len(counts), dtype=np.int32), counts)
    np.random.default_rng(seed).shuffle(ids)
    return ids.reshape(-1, 1).copy(), np.ones((ids.size, 1), dtype=np.float32)


@pytest.mark.parametrize("H,I", [(256, 256), (320, 192)])
def test_pair_gemms_every_last_tile(B, H, I):
    E = len(COUNTS)
    ids_np, _ = routing(COUNTS, seed=H + I)
    T = ids_np.shape[0]
    wl = wlm.custom("rem", T, E, 1, H, I, seed=H * 7 + I)
    x = wlm.make_x(wl, "cuda")
    W13, W2 = wlm.make_weights(wl, "cuda")
    p = B.Problem.make(T, E, 1, H, I, path=B.MOE_PATH_TILED, capacity=T + 64)
    offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(p.cap, dtype=torch.int32, device="cuda")
    inv = torch.empty(T, dtype=torch.int32, device="cuda")
    ws = torch.zeros(B.moe_workspace_size(p), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((p.cap, H), dtype=torch.bfloat16, device="cuda")
    ys = torch.full((p.cap, H), float("nan"), dtype=torch.float32, device="cuda")
    B.moe_dispatch(p, torch.from_numpy(ids_np).cuda(), offs, perm, inv, ws, x=x, x_sorted=xs)
    B.moe_expert_compute(p, xs, offs, W13, W2, ys, ws)
    torch.cuda.synchronize()
    assert B.moe_last_device_error(ws) == 0
    o = offs.cpu().numpy()
    assert np.array_equal(np.diff(o), COUNTS)
    n = int(o[-1])
    xs_np = wlm.bf16_bits(xs[:n])
    ref = np.zeros((n, H), dtype=np.float32)
    for e in range(E):
        a, b = int(o[e]), int(o[e + 1])
        if b > a:
            _, ref[a:b] = oracle.expert_rows(xs_np[a:b], wlm.bf16_bits(W13[e]), wlm.bf16_bits(W2[e]))
    for e in range(E):   # every expert on its own, so that a wrong last tile cannot hide in the average
        a, b = int(o[e]), int(o[e + 1])
        if b > a:
            assert_within_tolerance(ys[a:b].cpu().numpy(), ref[a:b], f"expert {e} ({COUNTS[e]} rows)")
    assert torch.isnan(ys[n:]).all()

    # the whole forward (fp16 y between the down GEMM and the combine)
    w = torch.ones((T, 1), dtype=torch.float32, device="cuda")
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    p2 = B.Problem.make(T, E, 1, H, I, path=B.MOE_PATH_TILED)
    ws2 = torch.zeros(B.moe_workspace_size(p2), dtype=torch.uint8, device="cuda")
    B.moe_forward(p2, x, torch.from_numpy(ids_np).cuda(), w, W13, W2, offs, perm, out, ws2)
    torch.cuda.synchronize()
    assert B.moe_last_device_error(ws2) == 0
    tokens = np.sort(np.random.default_rng(3).choice(T, 256, replace=False)).astype(np.int32)
    ref_acc, _, _ = oracle.moe_tokens(wlm.bf16_bits(x), ids_np, np.ones((T, 1), np.float32), wlm.bf16_bits(W13),
                                      wlm.bf16_bits(W2), tokens)
    assert_within_tolerance(wlm.bf16_bits(out)[tokens], ref_acc, "forward")
