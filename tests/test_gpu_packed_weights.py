"""Access-ordered PACKED weights (DeepGEMM PR #394, Summary: a weight layout in
the kernel's access order, bitwise-identical results to the row-major layout,
as in its Correctness section): the packed bytes follow the documented layout,
and every path gives bit-for-bit the same outputs from packed as from
row-major weights."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as wlm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from moe_routed_expert_routing_gb300.build import build
    build()
    from moe_routed_expert_routing_gb300 import binding
    return binding


def image(tile_rows: np.ndarray) -> np.ndarray:
    """[128 rows, 64 bf16] -> the 128-byte-swizzled shared-memory image: line r
    holds the row's 16-byte chunk c at position c XOR (r mod 8)."""
    chunks = tile_rows.reshape(128, 8, 8)
    out = np.empty_like(chunks)
    for r in range(128):
        for c in range(8):
            out[r, c ^ (r % 8)] = chunks[r, c]
    return out.reshape(-1)


def expected_packed(W13: np.ndarray, W2: np.ndarray):
    E, two_i, H = W13.shape
    I = two_i // 2
    p13 = []
    for e in range(E):
        for nt in range(I // 128):
            for kb in range(H // 64):
                cols = slice(kb * 64, kb * 64 + 64)
                p13.append(image(W13[e, nt * 128:nt * 128 + 128, cols]))
                p13.append(image(W13[e, I + nt * 128:I + nt * 128 + 128, cols]))
    p2 = []
    for e in range(E):
        for nt in range(H // 128):
            for kb in range(I // 64):
                p2.append(image(W2[e, nt * 128:nt * 128 + 128, kb * 64:kb * 64 + 64]))
    return np.concatenate(p13), np.concatenate(p2)


def test_packed_layout_matches_definition(B):
    wl = wlm.custom("pk", 4, 3, 2, 256, 256, seed=21)
    W13, W2 = wlm.make_weights(wl, "cuda")
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I)
    P13, P2 = B.moe_pack_weights(p, W13, W2)
    torch.cuda.synchronize()
    e13, e2 = expected_packed(wlm.bf16_bits(W13), wlm.bf16_bits(W2))
    assert np.array_equal(wlm.bf16_bits(P13).reshape(-1), e13)
    assert np.array_equal(wlm.bf16_bits(P2).reshape(-1), e2)


CASES = [
    # T, E, k, H, I, path
    (64, 8, 2, 256, 512, 1),
    (64, 8, 2, 256, 512, 2),
    (64, 8, 2, 256, 512, 3),
    (8, 24, 6, 1024, 768, 0),      # decode-like: M-small, split-K down GEMM
    (700, 3, 2, 512, 384, 1),      # CTA pairs, two pair tiles per expert
    (300, 16, 4, 768, 256, 0),     # single-CTA tiles
]


@pytest.mark.parametrize("case", CASES, ids=[f"T{c[0]}_E{c[1]}_p{c[5]}" for c in CASES])
def test_packed_weights_bitwise_equal(B, case):
    T, E, k, H, I, path = case
    wl = wlm.custom("pkf", T, E, k, H, I, seed=T + E)
    ids_np, w_np = wlm.make_routing(wl)
    x = wlm.make_x(wl, "cuda")
    W13, W2 = wlm.make_weights(wl, "cuda")
    ids = torch.from_numpy(ids_np).cuda()
    w = torch.from_numpy(w_np).cuda()
    outs = []
    for layout in (B.MOE_WEIGHTS_ROW_MAJOR, B.MOE_WEIGHTS_PACKED):
        p = B.Problem.make(T, E, k, H, I, path=path, weight_layout=layout)
        A13, A2 = (W13, W2) if layout == B.MOE_WEIGHTS_ROW_MAJOR else B.moe_pack_weights(p, W13, W2)
        bufs = B.Buffers(p)
        B.moe_forward(p, x, ids, w, A13, A2, bufs.expert_offsets, bufs.perm, bufs.out, bufs.ws)
        # the expert compute entry point on the same sorted batch
        ys = torch.full((p.cap, H), float("nan"), device="cuda")
        xs = torch.zeros((p.cap, H), dtype=torch.bfloat16, device="cuda")
        inv = torch.empty(T * k, dtype=torch.int32, device="cuda")
        B.moe_dispatch(p, ids, bufs.expert_offsets, bufs.perm, inv, bufs.ws, x=x, x_sorted=xs)
        B.moe_expert_compute(p, xs, bufs.expert_offsets, A13, A2, ys, bufs.ws)
        torch.cuda.synchronize()
        assert B.moe_last_device_error(bufs.ws) == 0
        n = int(bufs.expert_offsets[-1])
        outs.append((bufs.out.clone(), ys[:n].clone()))
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1].view(torch.int32), outs[1][1].view(torch.int32))
