"""GPU parity of moe_forward on the degenerate cases of the method, against the
oracle: no tokens, one expert (a dense gated MLP), every token on every expert,
an expert repeated inside one token, dropped and invalid slots, the largest
expert count, the smallest hidden/intermediate sizes and a wide top-k; each on
every GEMM path."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as wlm
from parity import assert_within_tolerance

pytestmark = pytest.mark.gpu

PATHS = [1, 2, 3]


@pytest.fixture(scope="module")
def B():
    from moe_routed_expert_routing_gb300.build import build
    build()
    from moe_routed_expert_routing_gb300 import binding
    return binding


def run_forward(B, p, x, ids_np, w_np, W13, W2, d_T=None):
    bufs = B.Buffers(p)
    bufs.out.fill_(7.0)
    B.moe_forward(p, x, torch.from_numpy(ids_np).cuda(), torch.from_numpy(w_np).cuda(), W13, W2,
                  bufs.expert_offsets, bufs.perm, bufs.out, bufs.ws, d_num_tokens=d_T)
    torch.cuda.synchronize()
    return bufs


def oracle_ref(x, ids_np, w_np, W13, W2):
    acc, out, bad = oracle.moe_tokens(wlm.bf16_bits(x), ids_np, w_np, wlm.bf16_bits(W13), wlm.bf16_bits(W2))
    return acc, bad


def make(T, E, k, H, I, seed, std=0.02):
    wl = wlm.custom("edge", T, E, k, H, I, seed=seed)
    x = wlm.make_x(wl, "cuda")
    W13, W2 = wlm.make_weights(wl, "cuda", std=std)
    return wl, x, W13, W2


@pytest.mark.parametrize("path", PATHS)
def test_zero_tokens_on_device(B, path):
    wl, x, W13, W2 = make(32, 8, 2, 256, 256, 1)
    ids_np, w_np = wlm.make_routing(wl)
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, path=path)
    d_T = torch.zeros(1, dtype=torch.int32, device="cuda")
    bufs = run_forward(B, p, x, ids_np, w_np, W13, W2, d_T=d_T)
    assert bufs.expert_offsets.cpu().numpy().tolist() == [0] * (wl.E + 1)
    assert torch.all(bufs.out == 7.0)                  # rows >= T are never written
    assert B.moe_last_device_error(bufs.ws) == 0


@pytest.mark.parametrize("path", PATHS)
def test_single_expert_is_a_dense_mlp(B, path):
    wl, x, W13, W2 = make(200, 1, 1, 512, 384, 2, std=0.04)
    ids_np = np.zeros((wl.T, 1), dtype=np.int32)
    w_np = np.ones((wl.T, 1), dtype=np.float32)
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, path=path)
    bufs = run_forward(B, p, x, ids_np, w_np, W13, W2)
    ref, _ = oracle_ref(x, ids_np, w_np, W13, W2)
    assert_within_tolerance(wlm.bf16_bits(bufs.out), ref, f"dense path {path}")
    # and against a dense gated MLP from torch matmuls (fp32 sums, bf16 activation)
    xf = x.float()
    h = (torch.nn.functional.silu(xf @ W13[0, :wl.I].float().T) * (xf @ W13[0, wl.I:].float().T)).to(torch.bfloat16)
    dense = (h.float() @ W2[0].float().T).cpu().numpy()
    assert_within_tolerance(wlm.bf16_bits(bufs.out), dense, f"dense torch path {path}")


@pytest.mark.parametrize("path", PATHS)
def test_every_token_on_every_expert(B, path):
    wl, x, W13, W2 = make(40, 4, 4, 256, 256, 3)
    ids_np = np.tile(np.arange(4, dtype=np.int32), (wl.T, 1))
    ids_np = np.ascontiguousarray(np.stack([np.random.default_rng(t).permutation(ids_np[t]) for t in range(wl.T)]))
    _, w_np = wlm.make_routing(wl)
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, path=path)
    bufs = run_forward(B, p, x, ids_np, w_np, W13, W2)
    ref, _ = oracle_ref(x, ids_np, w_np, W13, W2)
    assert_within_tolerance(wlm.bf16_bits(bufs.out), ref, f"k=E path {path}")


@pytest.mark.parametrize("path", PATHS)
def test_repeated_expert_dropped_and_invalid_slots(B, path):
    wl, x, W13, W2 = make(60, 8, 3, 256, 256, 4)
    ids_np, w_np = wlm.make_routing(wl)
    ids_np[0] = [5, 5, 1]          # the same expert twice in one token: two rows, both weighted
    ids_np[1] = [-1, 2, -1]        # dropped slots
    ids_np[2] = [3, 9, 0]          # 9 >= E: dropped and flagged
    w_np[2] = [0.5, 0.3, 0.2]
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, path=path)
    bufs = run_forward(B, p, x, ids_np, w_np, W13, W2)
    ref, bad = oracle_ref(x, ids_np, w_np, W13, W2)
    assert bad == 1
    assert B.moe_last_device_error(bufs.ws) & B.MOE_DEVERR_BAD_EXPERT_ID
    assert int(bufs.expert_offsets[-1]) == wl.R - 3
    assert_within_tolerance(wlm.bf16_bits(bufs.out), ref, f"dup/drop path {path}")


@pytest.mark.parametrize("path", PATHS)
def test_largest_expert_count(B, path):
    wl, x, W13, W2 = make(300, 1024, 4, 256, 128, 5)
    ids_np, w_np = wlm.make_routing(wl)
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, path=path)
    bufs = run_forward(B, p, x, ids_np, w_np, W13, W2)
    ref, _ = oracle_ref(x, ids_np, w_np, W13, W2)
    assert_within_tolerance(wlm.bf16_bits(bufs.out), ref, f"E=1024 path {path}")
    _, off, _, _, _ = oracle.dispatch(ids_np, wl.E)
    assert np.array_equal(bufs.expert_offsets.cpu().numpy(), off)


@pytest.mark.parametrize("path", PATHS)
def test_smallest_sizes_and_wide_topk(B, path):
    wl, x, W13, W2 = make(96, 32, 16, 256, 128, 6)
    ids_np, w_np = wlm.make_routing(wl)
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, path=path)
    bufs = run_forward(B, p, x, ids_np, w_np, W13, W2)
    ref, _ = oracle_ref(x, ids_np, w_np, W13, W2)
    assert_within_tolerance(wlm.bf16_bits(bufs.out), ref, f"H=256 I=128 k=16 path {path}")


def test_fp16_intermediate_y_range_is_reported(B):
    """moe_forward's tiled paths keep y in fp16: a down-GEMM output beyond
    +-65504 is clipped and MOE_DEVERR_Y_RANGE is set; in range, no flag."""
    T, E, k, H, I = 512, 8, 2, 256, 256          # a = 128 rows per expert: single-CTA tiles
    wl = wlm.custom("yrange", T, E, k, H, I, seed=13)
    ids_np, w_np = wlm.make_routing(wl)
    x = torch.ones((T, H), dtype=torch.bfloat16, device="cuda")
    W13 = torch.full((E, 2 * I, H), 0.01, dtype=torch.bfloat16, device="cuda")
    p = B.Problem.make(T, E, k, H, I)
    assert B.moe_resolve_path(p)[0] != 2
    for scale, flagged in [(1.0, False), (100.0, True)]:   # y ~ 256 * 6.1 * scale: 1.6e3 or 1.6e5
        W2 = torch.full((E, H, I), scale, dtype=torch.bfloat16, device="cuda")
        bufs = run_forward(B, p, x, ids_np, w_np, W13, W2)
        err = B.moe_last_device_error(bufs.ws)
        assert bool(err & B.MOE_DEVERR_Y_RANGE) == flagged, err
        assert torch.isfinite(bufs.out[:T].float()).all()


def test_binding_rejects_wrong_dtype_and_short_buffers(B):
    """The binding fails closed on CUDA tensors of the wrong dtype or extent,
    before any launch, and the buffers stay as they were."""
    p = B.Problem.make(16, 8, 2, 256, 128)
    wl = wlm.custom("bad", 16, 8, 2, 256, 128, seed=3)
    x = wlm.make_x(wl, "cuda")
    W13, W2 = wlm.make_weights(wl, "cuda")
    ids_np, w_np = wlm.make_routing(wl)
    ids = torch.from_numpy(ids_np).cuda()
    w = torch.from_numpy(w_np).cuda()
    bufs = B.Buffers(p)
    bufs.out.fill_(5.0)
    cases = [
        dict(topk_ids=ids.long()),                     # int64 ids
        dict(topk_weights=w.double()),                 # fp64 weights
        dict(x=x[:15]),                                # one token short
        dict(W2=W2[:7]),                               # one expert short
        dict(perm=bufs.perm[:-1]),                     # perm shorter than the capacity
    ]
    for bad in cases:
        args = dict(x=x, topk_ids=ids, topk_weights=w, W13=W13, W2=W2, expert_offsets=bufs.expert_offsets,
                    perm=bufs.perm, out=bufs.out, ws=bufs.ws)
        args.update(bad)
        with pytest.raises(ValueError):
            B.moe_forward(p, **args)
    torch.cuda.synchronize()
    assert torch.all(bufs.out == 5.0)
    assert B.moe_last_device_error(bufs.ws) == 0
