"""GPU parity at hidden and intermediate sizes that are multiples of 64 but not
of 128 or 256 (FlashInfer moe_ep page, Shape Coverage & Guardrails: hidden and
intermediate sizes that are multiples of 64, such as the 2880-wide
geometry). The last output-column tile of a GEMM then lies partly past H or
I: those columns are computed from neighbouring weight rows (or TMA zero
fill) and never stored. Every path and both decode forward forms run
against the oracle; a poisoned capacity tail shows that no store lands past
a row's last column."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as wlm
from parity import DeviceWorkload, assert_within_tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from moe_routed_expert_routing_gb300.build import build
    build()
    from moe_routed_expert_routing_gb300 import binding
    return binding


FORWARD = [
    # name, T, E, k, H, I  (H % 128 == 64 or I % 128 == 64)
    ("h448_i192", 512, 8, 2, 448, 192),
    ("h2880_i2880", 256, 16, 4, 2880, 2880),
    ("h320_i704", 160, 4, 2, 320, 704),
]


@pytest.mark.parametrize("case", FORWARD, ids=[c[0] for c in FORWARD])
@pytest.mark.parametrize("path", [0, 1, 2, 3])
def test_forward_multiple_of_64(B, case, path):
    name, T, E, k, H, I = case
    wl = wlm.custom(name, T, E, k, H, I, seed=H + I + T)
    dw = DeviceWorkload(wl)
    p = B.Problem.make(T, E, k, H, I, path=path)
    bufs = B.Buffers(p)
    B.moe_forward(p, dw.x, dw.ids, dw.w, dw.W13, dw.W2, bufs.expert_offsets, bufs.perm, bufs.out, bufs.ws)
    torch.cuda.synchronize()
    assert B.moe_last_device_error(bufs.ws) == 0
    tokens = wlm.token_subset(wl, 64 if T > 64 else 0)
    ref_acc, _ = dw.oracle_out(tokens)
    assert_within_tolerance(wlm.bf16_bits(bufs.out)[tokens], ref_acc, f"{name} path {path}")
    _, o_off, o_perm, _, _ = oracle.dispatch(dw.ids_np, E)
    assert np.array_equal(bufs.expert_offsets.cpu().numpy(), o_off)
    assert np.array_equal(bufs.perm.cpu().numpy()[: int(o_off[-1])], o_perm[: int(o_off[-1])])


DECODE = [
    # name, T, E, k, H, I: 16-row token tiles, both GEMMs in one persistent kernel
    ("dec_h448_i192", 8, 64, 4, 448, 192),    # I / 64 odd: the down GEMM keeps K whole
    ("dec_h448_i512", 4, 64, 4, 448, 512),    # the down GEMM splits K in two
    ("dec_h2880", 1, 32, 6, 2880, 2880),
]


@pytest.mark.parametrize("case", DECODE, ids=[c[0] for c in DECODE])
def test_decode_forms_multiple_of_64(B, case):
    name, T, E, k, H, I = case
    wl = wlm.custom(name, T, E, k, H, I, seed=H * 3 + I)
    dw = DeviceWorkload(wl)
    ref_acc, _ = dw.oracle_out()
    outs = {}
    for form in (B.MOE_FORWARD_SEPARATE, B.MOE_FORWARD_ONE_KERNEL):
        p = B.Problem.make(T, E, k, H, I, forward_form=form)
        assert B.moe_resolve_profile(p)["fused_mlp"] == 1
        bufs = B.Buffers(p)
        for _ in range(2):   # the second call reuses the counters the first one cleared
            B.moe_forward(p, dw.x, dw.ids, dw.w, dw.W13, dw.W2, bufs.expert_offsets, bufs.perm, bufs.out, bufs.ws)
        torch.cuda.synchronize()
        assert B.moe_last_device_error(bufs.ws) == 0
        assert_within_tolerance(wlm.bf16_bits(bufs.out), ref_acc, f"{name} form {form}")
        outs[form] = bufs.out.clone()
    assert torch.equal(outs[B.MOE_FORWARD_SEPARATE].view(torch.int16), outs[B.MOE_FORWARD_ONE_KERNEL].view(torch.int16))


COMPUTE = [
    # name, T, E, k, H, I, path
    ("ec_tiled", 300, 4, 2, 448, 192, 1),
    ("ec_tiled1", 300, 4, 2, 448, 192, 3),
    ("ec_small", 40, 32, 4, 448, 192, 2),
    ("ec_pair_h2880", 700, 3, 2, 2880, 320, 1),
]


@pytest.mark.parametrize("case", COMPUTE, ids=[c[0] for c in COMPUTE])
def test_expert_compute_multiple_of_64_and_no_store_past_the_row(B, case):
    """moe_expert_compute's y against the oracle's per-expert MLP; the rows of
    the capacity tail hold NaN before the call and must still hold it after:
    a store past column H of the last valid row would land there."""
    name, T, E, k, H, I, path = case
    wl = wlm.custom(name, T, E, k, H, I, seed=T + H)
    ids_np, _ = wlm.make_routing(wl)
    x = wlm.make_x(wl, "cuda")
    W13, W2 = wlm.make_weights(wl, "cuda")
    p = B.Problem.make(T, E, k, H, I, path=path, capacity=T * k + 64)
    offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(p.cap, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * k, dtype=torch.int32, device="cuda")
    ws = torch.zeros(B.moe_workspace_size(p), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((p.cap, H), dtype=torch.bfloat16, device="cuda")
    ys = torch.full((p.cap, H), float("nan"), dtype=torch.float32, device="cuda")
    B.moe_dispatch(p, torch.from_numpy(ids_np).cuda(), offs, perm, inv, ws, x=x, x_sorted=xs)
    B.moe_expert_compute(p, xs, offs, W13, W2, ys, ws)
    torch.cuda.synchronize()
    assert B.moe_last_device_error(ws) == 0
    o = offs.cpu().numpy()
    n = int(o[-1])
    xs_np = wlm.bf16_bits(xs[:n])
    ref = np.zeros((n, H), dtype=np.float32)
    for e in range(E):
        a, b = int(o[e]), int(o[e + 1])
        if b > a:
            _, ref[a:b] = oracle.expert_rows(xs_np[a:b], wlm.bf16_bits(W13[e]), wlm.bf16_bits(W2[e]))
    assert_within_tolerance(ys[:n].cpu().numpy(), ref, name)
    assert torch.isnan(ys[n:]).all()
