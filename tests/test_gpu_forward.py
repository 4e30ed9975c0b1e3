"""GPU parity of the whole routed expert execution (moe_forward) on the five
workloads against the oracle, plus the behaviours the TileOps page keeps
tests for (Review follow-up): capacity tail, graph replay, repeated-call
determinism, and a device-side token count behind a static capacity."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as wlm
from parity import DeviceWorkload, assert_within_tolerance, error_metrics

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from moe_routed_expert_routing_gb300.build import build
    build()
    from moe_routed_expert_routing_gb300 import binding
    return binding


def forward(B, p, dw, bufs=None, d_T=None, ids=None, w=None):
    bufs = bufs or B.Buffers(p)
    B.moe_forward(p, dw.x, dw.ids if ids is None else ids, dw.w if w is None else w, dw.W13, dw.W2,
                  bufs.expert_offsets, bufs.perm, bufs.out, bufs.ws, d_num_tokens=d_T)
    torch.cuda.synchronize()
    return bufs


@pytest.mark.parametrize("name", ["tiny", "decode1", "decode8", "small", "prefill", "large"])
def test_forward_matches_oracle(B, name):
    wl = wlm.WORKLOADS[name]
    dw = DeviceWorkload(wl)
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I)
    bufs = forward(B, p, dw)
    assert B.moe_last_device_error(bufs.ws) == 0
    tokens = wlm.token_subset(wl)
    ref_acc, _ = dw.oracle_out(tokens)
    got = wlm.bf16_bits(bufs.out)[tokens]
    m = assert_within_tolerance(got, ref_acc, name)
    print(name, m)


@pytest.mark.parametrize("name,path", [("tiny", 1), ("tiny", 2), ("tiny", 3), ("small", 1), ("small", 3),
                                       ("decode8", 1), ("large", 3)])
def test_forward_both_paths(B, name, path):
    wl = wlm.WORKLOADS[name]
    dw = DeviceWorkload(wl)
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, path=path)
    bufs = forward(B, p, dw)
    tokens = wlm.token_subset(wl, 64 if wl.T > 64 else 0)
    ref_acc, _ = dw.oracle_out(tokens)
    assert_within_tolerance(wlm.bf16_bits(bufs.out)[tokens], ref_acc, f"{name} path {path}")


@pytest.mark.parametrize("shape", [(512, 32, 4, 512, 256), (4, 64, 4, 512, 256)])
def test_repeated_forward_bit_exact(B, shape):
    """Repeated calls give identical bits (the second shape takes the split-K down GEMM)."""
    wl = wlm.custom("rep", *shape, seed=8)
    dw = DeviceWorkload(wl)
    for path in (1, 2, 3):
        p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, path=path)
        bufs = forward(B, p, dw)
        first = bufs.out.clone()
        for _ in range(3):
            forward(B, p, dw, bufs)
            assert torch.equal(first.view(torch.int16), bufs.out.view(torch.int16))


def test_capacity_tail_poison_does_not_leak(B):
    """capacity > T*k and a workspace full of NaN: out is unchanged (tail rows never read)."""
    wl = wlm.custom("cap", 100, 8, 2, 256, 256, seed=9)
    dw = DeviceWorkload(wl)
    p0 = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I)
    clean = forward(B, p0, dw).out.clone()
    for path in (1, 2, 3):
        p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, capacity=wl.R + 300, path=path)
        bufs = B.Buffers(p)
        bufs.ws.fill_(0xFF)                      # every bf16 in the sorted batches = NaN
        B.moe_clear_device_error(bufs.ws)
        forward(B, p, dw, bufs)
        assert torch.isfinite(bufs.out.float()).all()
        ref_acc, _ = dw.oracle_out()
        assert_within_tolerance(wlm.bf16_bits(bufs.out), ref_acc, f"capacity tail path {path}")
        if path == B.moe_resolve_path(p0)[0]:
            assert torch.equal(bufs.out.view(torch.int16), clean.view(torch.int16))


@pytest.mark.parametrize("shape", [(256, 16, 4, 512, 256), (1024, 8, 2, 512, 256)], ids=["tiled", "cta_pair"])
def test_graph_replay_new_routing_and_token_count(B, shape):
    """Capture one forward with a device token count; replay with new routing
    contents and other counts: bit-identical to eager calls (no host sync inside).
    Single-CTA tiles (64 rows per expert) and CTA-pair tiles (256)."""
    wl = wlm.custom("graph", *shape, seed=10)
    dw = DeviceWorkload(wl)
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I)
    bufs = B.Buffers(p)
    d_T = torch.tensor([wl.T], dtype=torch.int32, device="cuda")
    ids = dw.ids.clone()
    w = dw.w.clone()
    forward(B, p, dw, bufs, d_T=d_T, ids=ids, w=w)       # first call outside capture (function attributes)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            B.moe_forward(p, dw.x, ids, w, dw.W13, dw.W2, bufs.expert_offsets, bufs.perm, bufs.out, bufs.ws,
                          d_num_tokens=d_T, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for seed, T_dev in [(101, wl.T), (102, wl.T // 2), (103, 1)]:
        ids_np, w_np = wlm.make_routing(wl, seed=seed)
        ids.copy_(torch.from_numpy(ids_np))
        w.copy_(torch.from_numpy(w_np))
        d_T.fill_(T_dev)
        bufs.out.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        got = bufs.out[:T_dev].clone()
        eager = B.Buffers(p)
        eager.out.fill_(0)
        forward(B, p, dw, eager, d_T=d_T, ids=ids, w=w)
        assert torch.equal(got.view(torch.int16), eager.out[:T_dev].view(torch.int16))
        tokens = np.arange(T_dev, dtype=np.int32)
        ref_acc, _ = dw.oracle_out(tokens, ids_np=ids_np, w_np=w_np)
        assert_within_tolerance(wlm.bf16_bits(got), ref_acc, f"graph replay T={T_dev}")


def test_prefill_dynamic_capacity_sampled(B):
    """Prefill shape, graph-style static capacity T_max*k with device T in {2048, 1024, 1}."""
    wl = wlm.WORKLOADS["prefill"]
    dw = DeviceWorkload(wl)
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I)
    bufs = B.Buffers(p)
    d_T = torch.zeros(1, dtype=torch.int32, device="cuda")
    for T_dev in (1024, 1):
        d_T.fill_(T_dev)
        forward(B, p, dw, bufs, d_T=d_T)
        off = bufs.expert_offsets.cpu().numpy()
        assert off[-1] == T_dev * wl.k
        tokens = np.sort(np.random.default_rng(T_dev).choice(T_dev, min(T_dev, 32), replace=False)).astype(np.int32)
        ids_np = dw.ids_np[:T_dev]
        ref_acc, _ = dw.oracle_out(tokens, ids_np=ids_np, w_np=dw.w_np[:T_dev])
        m = error_metrics(wlm.bf16_bits(bufs.out)[tokens], ref_acc)
        assert m["max_err_beyond_output_rounding"] <= m["bound"] and m["mean_rel_err"] <= 5e-3, m


def test_launch_profile_table(B):
    """The static profile follows from the shape alone (a = T_max*k/E rows per expert)."""
    P = B.Problem.make
    dec1 = B.moe_resolve_profile(P(1, 384, 6, 7168, 3072))
    # one token at E=384: 336 full-K down units; 4 K parts (1344 units) fill the waves best;
    # AUTO keeps three kernels (measured faster than one with 4 K parts)
    assert dec1 == dict(path=2, tile_rows=16, down_split_k=4, pdl=1, fused_gather=1, cta_pair=0, fused_mlp=1,
                        megakernel=0, kernel_launches=3)
    assert B.moe_resolve_profile(P(1, 384, 6, 7168, 3072, forward_form=B.MOE_FORWARD_ONE_KERNEL))["megakernel"] == 1
    dec8 = B.moe_resolve_profile(P(8, 384, 6, 7168, 3072))
    assert dec8 == dict(path=2, tile_rows=16, down_split_k=1, pdl=1, fused_gather=1, cta_pair=0, fused_mlp=1,
                        megakernel=0, kernel_launches=3)
    assert B.moe_resolve_profile(P(8, 384, 6, 7168, 3072, forward_form=B.MOE_FORWARD_ONE_KERNEL))["megakernel"] == 1
    # MXFP8 weights: AUTO keeps three kernels at T=1 (measured faster); one kernel on request
    assert B.moe_resolve_profile(P(1, 384, 6, 7168, 3072, weight_layout=B.MOE_WEIGHTS_MXFP8))["megakernel"] == 0
    assert B.moe_resolve_profile(P(1, 384, 6, 7168, 3072, weight_layout=B.MOE_WEIGHTS_MXFP8,
                                   forward_form=B.MOE_FORWARD_ONE_KERNEL))["megakernel"] == 1
    assert B.moe_resolve_profile(P(1, 384, 6, 7168, 3072, forward_form=B.MOE_FORWARD_SEPARATE))["megakernel"] == 0
    with pytest.raises(B.MoeError) as ei:      # not decode-size: one kernel is refused, not ignored
        B.moe_resolve_profile(P(128, 256, 8, 7168, 2048, forward_form=B.MOE_FORWARD_ONE_KERNEL))
    assert ei.value.status == 5
    small = B.moe_resolve_profile(P(128, 256, 8, 7168, 2048))
    assert small["path"] == 2 and small["tile_rows"] == 32 and small["down_split_k"] == 1 and small["fused_mlp"] == 0
    assert small["megakernel"] == 0 and small["kernel_launches"] == 4    # dispatch, 2 GEMMs, combine
    prefill = B.moe_resolve_profile(P(2048, 384, 6, 7168, 3072))
    assert prefill == dict(path=3, tile_rows=128, down_split_k=1, pdl=0, fused_gather=0, cta_pair=0, fused_mlp=0,
                           megakernel=0, kernel_launches=7)
    large = B.moe_resolve_profile(P(8192, 128, 8, 4096, 1536))
    assert large == dict(path=1, tile_rows=128, down_split_k=1, pdl=0, fused_gather=0, cta_pair=1, fused_mlp=0,
                         megakernel=0, kernel_launches=7)
    # the boundaries of the rule: M-small up to a = 8, single-CTA tiles below a = 128, CTA pairs from it
    assert B.moe_resolve_profile(P(512, 384, 6, 7168, 3072))["path"] == 2          # a = 8
    assert B.moe_resolve_profile(P(768, 384, 6, 7168, 3072))["path"] == 3          # a = 12
    assert B.moe_resolve_profile(P(6144, 384, 6, 7168, 3072))["path"] == 3         # a = 96
    assert B.moe_resolve_profile(P(8192, 384, 6, 7168, 3072))["path"] == 1         # a = 128
    # 16-row tiles whose shared-memory dispatch tables do not fit: fused GEMMs, separate dispatch and combine
    wide = B.moe_resolve_profile(P(256, 1024, 8, 512, 256))
    assert wide["fused_mlp"] == 1 and wide["megakernel"] == 0 and wide["kernel_launches"] == 5   # 3 dispatch


@pytest.mark.parametrize("form", [1, 2], ids=["separate", "one_kernel"])
def test_fused_decode_kernel_graph_replay_token_counts(B, form):
    """Decode-size batches run both GEMMs as one persistent kernel with per-expert
    readiness counts (and, in the one-kernel form, dispatch and combine too):
    captured once, replayed with T in {8, 3, 1, 0}, every replay equals an
    eager call bit for bit and the oracle within tolerance."""
    wl = wlm.custom("fusedgraph", 8, 64, 4, 512, 256, seed=44)
    dw = DeviceWorkload(wl)
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, forward_form=form)
    assert B.moe_resolve_profile(p)["fused_mlp"] == 1
    assert B.moe_resolve_profile(p)["megakernel"] == (form == 2)
    bufs = B.Buffers(p)
    d_T = torch.tensor([wl.T], dtype=torch.int32, device="cuda")
    forward(B, p, dw, bufs, d_T=d_T)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            B.moe_forward(p, dw.x, dw.ids, dw.w, dw.W13, dw.W2, bufs.expert_offsets, bufs.perm, bufs.out, bufs.ws,
                          d_num_tokens=d_T, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for T_dev in (8, 3, 1, 0):
        d_T.fill_(T_dev)
        bufs.out.fill_(5.0)
        g.replay()
        torch.cuda.synchronize()
        assert B.moe_last_device_error(bufs.ws) == 0
        assert torch.all(bufs.out[T_dev:] == 5.0)
        if T_dev == 0:
            continue
        eager = B.Buffers(p)
        forward(B, p, dw, eager, d_T=d_T)
        assert torch.equal(bufs.out[:T_dev].view(torch.int16), eager.out[:T_dev].view(torch.int16))
        ref_acc, _ = dw.oracle_out(np.arange(T_dev, dtype=np.int32))
        assert_within_tolerance(wlm.bf16_bits(bufs.out[:T_dev]), ref_acc, f"fused T={T_dev}")


def _separate_entry_points(B, p, dw, d_T=None):
    """dispatch -> expert compute -> combine through the three separate calls."""
    bufs = B.Buffers(p)
    B.moe_dispatch(p, dw.ids, bufs.expert_offsets, bufs.perm, bufs.inv, bufs.ws, x=dw.x, x_sorted=bufs.x_sorted,
                   d_num_tokens=d_T)
    B.moe_expert_compute(p, bufs.x_sorted, bufs.expert_offsets, dw.W13, dw.W2, bufs.y_sorted, bufs.ws)
    bufs.out.fill_(3.0)
    B.moe_combine(p, bufs.y_sorted, bufs.inv, dw.w, bufs.out, d_num_tokens=d_T)
    torch.cuda.synchronize()
    return bufs


# (T, E, k, H, I), down GEMM K parts (made of 128-wide K blocks): one token
# (4 parts; 2 where I holds two blocks), a decode batch (unsplit), a wide
# top-k (2 parts), I not a multiple of 128 (unsplit)
MEGA_SHAPES = [((1, 64, 6, 512, 512), 4), ((1, 64, 4, 512, 256), 2), ((8, 64, 4, 4096, 256), 1),
               ((24, 256, 16, 256, 256), 2), ((1, 64, 4, 512, 192), 1)]


@pytest.mark.parametrize("shape,parts", MEGA_SHAPES, ids=["T1_split4", "T1_split2", "T8", "k16", "T1_i192"])
def test_megakernel_equals_separate_entry_points(B, shape, parts):
    """The one-kernel forward gives the same bits as dispatch + expert compute +
    combine launched separately (same GEMM arithmetic, the down GEMM's K parts
    summed in the same order, same combine order), and the same expert_offsets
    and perm; the three-kernel forward too."""
    wl = wlm.custom("mega", *shape, seed=sum(shape))
    dw = DeviceWorkload(wl)
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, forward_form=B.MOE_FORWARD_ONE_KERNEL)
    prof = B.moe_resolve_profile(p)
    assert prof["megakernel"] == 1 and prof["kernel_launches"] == 1 and prof["down_split_k"] == parts
    got = forward(B, p, dw)
    assert B.moe_last_device_error(got.ws) == 0
    ref = _separate_entry_points(B, p, dw)
    assert torch.equal(got.expert_offsets, ref.expert_offsets)
    n = int(ref.expert_offsets[-1])
    assert torch.equal(got.perm[:n], ref.perm[:n])
    assert torch.equal(got.out.view(torch.int16), ref.out.view(torch.int16))
    three = forward(B, B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, forward_form=B.MOE_FORWARD_SEPARATE), dw)
    assert torch.equal(three.out.view(torch.int16), ref.out.view(torch.int16))
    ref_acc, _ = dw.oracle_out()
    assert_within_tolerance(wlm.bf16_bits(got.out), ref_acc, f"megakernel {shape}")


# error word, per-expert readiness counts, the fused kernel's three GPU-wide
# counters and the separate grouped GEMMs' two (units handed out, CTAs at the tail)
HEADER_BYTES = 256 + 4 * (1024 + 5)


@pytest.mark.parametrize("path", [1, 2, 3], ids=["pair", "small_m", "tiled_1cta"])
def test_unit_counts_return_to_zero(B, path):
    """GEMMs with more units than CTAs take units from GPU-wide counts in the
    workspace header (the M-small down GEMM and the single-CTA tiled GEMMs);
    after every call of moe_forward and of moe_expert_compute the header is
    zero again, repeated calls are bit-identical, and the output matches the
    oracle on a token subset."""
    wl = wlm.custom("units", 1024, 16, 4, 1024, 1024, seed=71)
    dw = DeviceWorkload(wl)
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, path=path)
    bufs = B.Buffers(p)
    first = None
    for _ in range(3):
        forward(B, p, dw, bufs)
        assert B.moe_last_device_error(bufs.ws) == 0
        assert int(bufs.ws[:HEADER_BYTES].count_nonzero()) == 0
        if first is None:
            first = bufs.out.clone()
        assert torch.equal(first.view(torch.int16), bufs.out.view(torch.int16))
    tokens = wlm.token_subset(wl, 64)
    ref_acc, _ = dw.oracle_out(tokens)
    assert_within_tolerance(wlm.bf16_bits(first)[tokens], ref_acc, f"path {path}")
    # moe_expert_compute on the same workspace, twice
    cap = p.cap
    offs = torch.empty(wl.E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(cap, dtype=torch.int32, device="cuda")
    inv = torch.empty(wl.T * wl.k, dtype=torch.int32, device="cuda")
    xs = torch.zeros((cap, wl.H), dtype=torch.bfloat16, device="cuda")
    B.moe_dispatch(p, dw.ids, offs, perm, inv, bufs.ws, x=dw.x, x_sorted=xs)
    ys = []
    for _ in range(2):
        y = torch.zeros((cap, wl.H), dtype=torch.float32, device="cuda")
        B.moe_expert_compute(p, xs, offs, dw.W13, dw.W2, y, bufs.ws)
        torch.cuda.synchronize()
        assert B.moe_last_device_error(bufs.ws) == 0
        assert int(bufs.ws[:HEADER_BYTES].count_nonzero()) == 0
        ys.append(y)
    assert torch.equal(ys[0], ys[1])


def test_megakernel_tail_clears_its_counters(B):
    """Workspace header after every call: error word, readiness counts and the
    two GPU-wide counters all back at zero; repeated calls bit-identical. A
    workspace of garbage is readied by moe_clear_device_error."""
    wl = wlm.custom("megatail", 8, 128, 6, 512, 256, seed=61)
    dw = DeviceWorkload(wl)
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, forward_form=B.MOE_FORWARD_ONE_KERNEL)
    assert B.moe_resolve_profile(p)["megakernel"] == 1
    bufs = B.Buffers(p)
    header = HEADER_BYTES
    first = None
    for _ in range(4):
        forward(B, p, dw, bufs)
        assert int(bufs.ws[:header].count_nonzero()) == 0
        if first is None:
            first = bufs.out.clone()
        assert torch.equal(first.view(torch.int16), bufs.out.view(torch.int16))
    bufs.ws.fill_(0x5A)
    B.moe_clear_device_error(bufs.ws)
    forward(B, p, dw, bufs)
    assert B.moe_last_device_error(bufs.ws) == 0
    assert torch.equal(first.view(torch.int16), bufs.out.view(torch.int16))
    assert int(bufs.ws[:header].count_nonzero()) == 0


def test_megakernel_dropped_invalid_and_repeated_slots(B):
    """Degenerate routing inside the one-kernel forward: a repeated expert in
    one token, dropped slots (-1), an out-of-range id (dropped and flagged),
    and a device token count below T_max (rows >= T untouched)."""
    wl = wlm.custom("megaedge", 12, 64, 4, 512, 256, seed=62)
    dw = DeviceWorkload(wl)
    ids_np, w_np = dw.ids_np.copy(), dw.w_np.copy()
    ids_np[0] = [7, 7, 1, 2]
    ids_np[1] = [-1, 3, -1, 4]
    ids_np[2] = [5, 99, 6, 0]
    ids = torch.from_numpy(ids_np).cuda()
    w = torch.from_numpy(w_np).cuda()
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, forward_form=B.MOE_FORWARD_ONE_KERNEL)
    assert B.moe_resolve_profile(p)["megakernel"] == 1
    d_T = torch.tensor([10], dtype=torch.int32, device="cuda")
    bufs = B.Buffers(p)
    bufs.out.fill_(9.0)
    forward(B, p, dw, bufs, d_T=d_T, ids=ids, w=w)
    assert B.moe_last_device_error(bufs.ws) & B.MOE_DEVERR_BAD_EXPERT_ID
    assert torch.all(bufs.out[10:] == 9.0)
    valid = int(np.count_nonzero((ids_np[:10] >= 0) & (ids_np[:10] < wl.E)))
    assert int(bufs.expert_offsets[-1]) == valid
    tokens = np.arange(10, dtype=np.int32)
    ref_acc, _ = dw.oracle_out(tokens, ids_np=ids_np, w_np=w_np)
    assert_within_tolerance(wlm.bf16_bits(bufs.out[:10]), ref_acc, "megakernel degenerate routing")


@pytest.mark.parametrize("name", ["prefill", "large"])
def test_prefill_graph_replay_device_token_counts(B, name):
    """Prefill shape (single-CTA tiles) and large shape (CTA-pair tiles)
    captured once as a CUDA graph at T_max (static capacity T_max*k), replayed
    with device T in {T_max, T_max/2, 1}: each replay equals an eager call bit
    for bit, leaves rows >= T untouched, and matches the oracle on sampled
    tokens."""
    wl = wlm.WORKLOADS[name]
    dw = DeviceWorkload(wl)
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I)
    bufs = B.Buffers(p)
    d_T = torch.tensor([wl.T], dtype=torch.int32, device="cuda")
    forward(B, p, dw, bufs, d_T=d_T)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            B.moe_forward(p, dw.x, dw.ids, dw.w, dw.W13, dw.W2, bufs.expert_offsets, bufs.perm, bufs.out, bufs.ws,
                          d_num_tokens=d_T, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    eager = B.Buffers(p)
    for T_dev in (wl.T, wl.T // 2, 1):
        d_T.fill_(T_dev)
        bufs.out.fill_(2.0)
        g.replay()
        torch.cuda.synchronize()
        assert B.moe_last_device_error(bufs.ws) == 0
        assert int(bufs.expert_offsets[-1]) == T_dev * wl.k
        assert torch.all(bufs.out[T_dev:] == 2.0)
        forward(B, p, dw, eager, d_T=d_T)
        assert torch.equal(bufs.out[:T_dev].view(torch.int16), eager.out[:T_dev].view(torch.int16))
        tokens = np.sort(np.random.default_rng(T_dev + 7).choice(T_dev, min(T_dev, 32), replace=False)).astype(np.int32)
        ref_acc, _ = dw.oracle_out(tokens, ids_np=dw.ids_np[:T_dev], w_np=dw.w_np[:T_dev])
        assert_within_tolerance(wlm.bf16_bits(bufs.out)[tokens], ref_acc, f"{name} graph T={T_dev}")
