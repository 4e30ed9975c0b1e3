"""MXFP8 expert weights (OCP MX: E4M3 codes, one E8M0 scale per 32 K-elements;
the pages' MXFP8 path, FlashInfer moe_ep page PR #3980): the GPU quantizer
against the oracle's, byte for byte, and moe_forward on MXFP8 weights against
the bf16 forward on the dequantized weights (bit for bit: the expansion to
bf16 is exact and the K order of the MMAs is the same) and against the
oracle. Every M-small tile height, split-K, and the one-kernel form."""
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


def untile_scales(sc_tiled: np.ndarray, rows: int, K: int) -> np.ndarray:
    """Scale blocks (128-row tile, 128-wide K block, row, sub-block) -> row-major [rows, K/32]."""
    t = sc_tiled.reshape(rows // 128, K // 128, 128, 4)
    return t.transpose(0, 2, 1, 3).reshape(rows, K // 32)


def split_mx(buf: torch.Tensor, rows: int, K: int):
    h = buf.cpu().numpy()
    return h[: rows * K].reshape(rows, K), untile_scales(h[rows * K:], rows, K)


def quantized(B, p, W13, W2):
    W13_mx, W2_mx = B.moe_quantize_weights(p, W13, W2)
    torch.cuda.synchronize()
    E, H, I = p.E, p.H, p.I
    q13, s13 = split_mx(W13_mx, E * 2 * I, H)
    q2, s2 = split_mx(W2_mx, E * H, I)
    return W13_mx, W2_mx, (q13, s13), (q2, s2)


def dequantized_device(q, s, shape):
    return torch.from_numpy(oracle.mx_dequantize(q, s).view(np.int16).reshape(shape)).view(torch.bfloat16).cuda()


def test_weight_bytes(B):
    p = B.Problem.make(8, 384, 6, 7168, 3072)
    b13, b2 = B.moe_weight_bytes(p, B.MOE_WEIGHTS_MXFP8)
    assert b13 == 384 * 6144 * 7168 * 33 // 32 and b2 == 384 * 7168 * 3072 * 33 // 32
    assert B.moe_weight_bytes(p, B.MOE_WEIGHTS_ROW_MAJOR) == (384 * 6144 * 7168 * 2, 384 * 7168 * 3072 * 2)


def test_quantizer_matches_oracle_bytes(B):
    wl = wlm.custom("mxq", 8, 4, 2, 512, 256, seed=21)
    W13, W2 = wlm.make_weights(wl, "cuda", std=0.02)
    # special blocks: zeros, one large outlier (saturation of its neighbours is not
    # possible: the outlier sets the scale), tiny values, exact grid values
    W13[0, 0, :32] = 0
    W13[1, 5, 64:96] = torch.linspace(-3.0, 3.0, 32)
    W13[2, 7, 128:160] = 1e-6
    W2[3, 1, :32] = torch.tensor([448.0 * 2.0 ** -10] + [0.0] * 31)
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I)
    _, _, (q13, s13), (q2, s2) = quantized(B, p, W13, W2)
    oq13, os13 = oracle.mx_quantize(wlm.bf16_bits(W13).reshape(-1, wl.H))
    oq2, os2 = oracle.mx_quantize(wlm.bf16_bits(W2).reshape(-1, wl.I))
    assert np.array_equal(s13, os13) and np.array_equal(s2, os2)
    assert np.array_equal(q13, oq13), np.argwhere(q13 != oq13)[:5]
    assert np.array_equal(q2, oq2), np.argwhere(q2 != oq2)[:5]


def test_quantizer_matches_oracle_decode_shape_sampled(B):
    """The decode layer shape (E=384, H=7168, I=3072): two experts compared in full."""
    wl = wlm.WORKLOADS["decode8"]
    W13, W2 = wlm.make_weights(wl, "cuda")
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I)
    W13_mx, W2_mx = B.moe_quantize_weights(p, W13, W2)
    torch.cuda.synchronize()
    h13 = W13_mx.cpu().numpy()
    h2 = W2_mx.cpu().numpy()
    r13, r2 = wl.E * 2 * wl.I, wl.E * wl.H
    s13 = untile_scales(h13[r13 * wl.H:], r13, wl.H)
    s2 = untile_scales(h2[r2 * wl.I:], r2, wl.I)
    for e in (0, 383):
        oq, os_ = oracle.mx_quantize(wlm.bf16_bits(W13[e]))
        rows = slice(e * 2 * wl.I, (e + 1) * 2 * wl.I)
        assert np.array_equal(h13[: r13 * wl.H].reshape(r13, wl.H)[rows], oq)
        assert np.array_equal(s13[rows], os_)
        oq, os_ = oracle.mx_quantize(wlm.bf16_bits(W2[e]))
        rows = slice(e * wl.H, (e + 1) * wl.H)
        assert np.array_equal(h2[: r2 * wl.I].reshape(r2, wl.I)[rows], oq)
        assert np.array_equal(s2[rows], os_)


# (T, E, k, H, I, form): tile 16 with the down GEMM in 2 K parts (AUTO: three
# kernels), in 4 K parts (three kernels, then one), tile 16 unsplit, tile 16
# unsplit as one kernel, tile 32, tile 64, tile 64 with several token tiles
# per expert (128 rows per expert: bf16 weights would take a tiled path there,
# MXFP8 stays on the M-small path at every batch size)
CASES = [(1, 64, 4, 512, 256, 0), (1, 64, 6, 512, 512, 0), (1, 64, 6, 512, 512, 2), (8, 64, 4, 4096, 256, 0),
         (8, 64, 4, 4096, 256, 2), (64, 32, 4, 512, 384, 0), (100, 32, 4, 512, 256, 0), (512, 16, 4, 512, 512, 0)]


@pytest.mark.parametrize("case", CASES, ids=["t16_split2", "t16_split4", "t16_split4_one_kernel", "t16",
                                             "t16_one_kernel", "t32", "t64", "t64_many_tiles"])
def test_mxfp8_forward_equals_bf16_forward_on_dequantized(B, case):
    T, E, k, H, I, form = case
    wl = wlm.custom("mxf", T, E, k, H, I, seed=T + E + H)
    x = wlm.make_x(wl, "cuda")
    W13, W2 = wlm.make_weights(wl, "cuda")
    ids_np, w_np = wlm.make_routing(wl)
    ids, w = torch.from_numpy(ids_np).cuda(), torch.from_numpy(w_np).cuda()
    p_mx = B.Problem.make(T, E, k, H, I, weight_layout=B.MOE_WEIGHTS_MXFP8, forward_form=form)
    prof = B.moe_resolve_profile(p_mx)
    assert prof["path"] == 2 and prof["fused_mlp"] == 1
    # MXFP8 and bf16 weights split the down GEMM's K alike (128-wide blocks)
    assert prof["down_split_k"] == B.moe_resolve_profile(B.Problem.make(T, E, k, H, I, forward_form=form, path=2))[
        "down_split_k"]
    if I == 512 and T == 1:
        assert prof["down_split_k"] == 4
    W13_mx, W2_mx, (q13, s13), (q2, s2) = quantized(B, p_mx, W13, W2)
    W13_d = dequantized_device(q13, s13, W13.shape)
    W2_d = dequantized_device(q2, s2, W2.shape)
    outs = []
    for p, a, b in [(p_mx, W13_mx, W2_mx), (B.Problem.make(T, E, k, H, I, forward_form=form, path=2), W13_d, W2_d)]:
        bufs = B.Buffers(p)
        B.moe_forward(p, x, ids, w, a, b, bufs.expert_offsets, bufs.perm, bufs.out, bufs.ws)
        torch.cuda.synchronize()
        assert B.moe_last_device_error(bufs.ws) == 0
        outs.append(bufs.out.clone())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    ref_acc, _, _ = oracle.moe_tokens(wlm.bf16_bits(x), ids_np, w_np, wlm.bf16_bits(W13_d), wlm.bf16_bits(W2_d))
    assert_within_tolerance(wlm.bf16_bits(outs[0]), ref_acc, f"mxfp8 {case}")


def test_mxfp8_forward_scale_extremes(B):
    """Blocks at the ends of the scale range the expansion handles: maxima >= 2^16
    (scale exponent e > 7, expanded with two bf16 multiplies), a block at 2^-110
    (e = -118, the smallest the format note allows), blocks whose small entries
    quantize to E4M3 subnormal codes, a zero
    block and signed zeros; in both GEMMs of touched experts. The forward on the
    MXFP8 weights equals the bf16 forward on the dequantized weights bit for bit."""
    T, E, k, H, I = 8, 8, 2, 512, 256
    wl = wlm.custom("mxext", T, E, k, H, I, seed=57)
    x = wlm.make_x(wl, "cuda")
    W13, W2 = wlm.make_weights(wl, "cuda")
    ids_np, w_np = wlm.make_routing(wl)
    ids_np[0] = [0, 1]
    ids_np[1] = [1, 2]
    ids, w = torch.from_numpy(ids_np).cuda(), torch.from_numpy(w_np).cuda()
    W13[0, 3, :32] *= 2.0 ** 24                     # gate row: max ~2^19, e = 11
    W13[1, I + 9, 64:96] *= 2.0 ** 17               # up row: e around 4..5, and one block pushed above 2^16
    W13[1, I + 9, 64] = 70000.0
    # e = -118; 2^-126 and 2^-127 quantize to E4M3 subnormal codes whose values are a
    # bf16 normal and a bf16 subnormal
    W13[2, 5, 32:64] = torch.tensor([2.0 ** -110, -(2.0 ** -113), 2.0 ** -126, -(2.0 ** -127)] + [2.0 ** -118] * 28)
    W13[0, 7, 96:128] = torch.tensor([1.0, -1e-5, 3e-6, -2e-6] + [0.0] * 14 + [-0.0] * 14)   # subnormal codes
    W2[0, 11, :32] *= 2.0 ** 24                     # down GEMM: e > 7 as well
    W2[1, 2, 32:64] = torch.tensor([-0.5, 1e-5] + [0.0] * 30)
    W2[2, 4, :32] = 0
    p_mx = B.Problem.make(T, E, k, H, I, weight_layout=B.MOE_WEIGHTS_MXFP8)
    W13_mx, W2_mx, (q13, s13), (q2, s2) = quantized(B, p_mx, W13, W2)
    assert s13.max() > 127 + 7 and s2.max() > 127 + 7 and s13.min() == 127 - 118
    assert np.any((q13 & 0x78) == 0) and np.any(((q13 & 0x78) == 0) & ((q13 & 0x07) != 0))   # subnormal codes
    W13_d = dequantized_device(q13, s13, W13.shape)
    W2_d = dequantized_device(q2, s2, W2.shape)
    outs = []
    for p, a, b in [(p_mx, W13_mx, W2_mx), (B.Problem.make(T, E, k, H, I), W13_d, W2_d)]:
        bufs = B.Buffers(p)
        B.moe_forward(p, x, ids, w, a, b, bufs.expert_offsets, bufs.perm, bufs.out, bufs.ws)
        torch.cuda.synchronize()
        assert B.moe_last_device_error(bufs.ws) == 0
        outs.append(bufs.out.clone())
    assert torch.isfinite(outs[0].float()).all()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_mxfp8_refused_outside_the_m_small_path(B):
    """AUTO takes the M-small path for MXFP8 weights at any batch size; a tiled
    path asked for explicitly, and moe_expert_compute, refuse the layout."""
    auto = B.moe_resolve_profile(B.Problem.make(2048, 384, 6, 7168, 3072, weight_layout=B.MOE_WEIGHTS_MXFP8))
    assert auto["path"] == 2 and auto["tile_rows"] == 64 and auto["fused_mlp"] == 1
    # 64-row token tiles read a sorted copy of x (a gather kernel first): dispatch (3), gather, GEMMs, combine
    assert auto["fused_gather"] == 0 and auto["kernel_launches"] == 6
    # decode-size MXFP8 batches read the sorted copy too (dispatch, gather, GEMMs, combine); the
    # one-kernel form gathers inside its CTAs
    dec = B.moe_resolve_profile(B.Problem.make(8, 384, 6, 7168, 3072, weight_layout=B.MOE_WEIGHTS_MXFP8))
    assert dec["tile_rows"] == 16 and dec["fused_gather"] == 0 and dec["kernel_launches"] == 4
    one = B.moe_resolve_profile(B.Problem.make(8, 384, 6, 7168, 3072, weight_layout=B.MOE_WEIGHTS_MXFP8,
                                               forward_form=B.MOE_FORWARD_ONE_KERNEL))
    assert one["megakernel"] == 1 and one["fused_gather"] == 1 and one["kernel_launches"] == 1
    for path in (1, 3):
        p = B.Problem.make(2048, 384, 6, 7168, 3072, weight_layout=B.MOE_WEIGHTS_MXFP8, path=path)
        with pytest.raises(B.MoeError) as ei:
            B.moe_resolve_profile(p)
        assert ei.value.status == 5
    q = B.Problem.make(8, 64, 4, 512, 256, weight_layout=B.MOE_WEIGHTS_MXFP8)
    bufs = B.Buffers(q)
    W = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.MoeError) as ei:
        B.moe_expert_compute(q, bufs.x_sorted, bufs.expert_offsets, W, W, bufs.y_sorted, bufs.ws)
    assert ei.value.status == 5


def test_mxfp8_degenerate_routing_and_graph_replay(B):
    """MXFP8 weights under the edge cases of the method: a repeated expert in
    one token, dropped (-1) and out-of-range ids, and a device token count
    replayed from one captured graph with T in {12, 5, 1, 0} (rows >= T
    untouched); every replay against an eager call (bit for bit) and the
    oracle on the dequantized weights."""
    T, E, k, H, I = 12, 64, 4, 512, 256
    wl = wlm.custom("mxedge", T, E, k, H, I, seed=91)
    x = wlm.make_x(wl, "cuda")
    W13, W2 = wlm.make_weights(wl, "cuda")
    ids_np, w_np = wlm.make_routing(wl)
    ids_np[0] = [7, 7, 1, 2]
    ids_np[1] = [-1, 3, -1, 4]
    ids_np[2] = [5, 99, 6, 0]
    ids, w = torch.from_numpy(ids_np).cuda(), torch.from_numpy(w_np).cuda()
    for form in (1, 2):
        p = B.Problem.make(T, E, k, H, I, weight_layout=B.MOE_WEIGHTS_MXFP8, forward_form=form)
        W13_mx, W2_mx, (q13, s13), (q2, s2) = quantized(B, p, W13, W2)
        W13_d = oracle.mx_dequantize(q13, s13).view(np.uint16).reshape(W13.shape)
        W2_d = oracle.mx_dequantize(q2, s2).view(np.uint16).reshape(W2.shape)
        bufs = B.Buffers(p)
        d_T = torch.tensor([T], dtype=torch.int32, device="cuda")
        B.moe_forward(p, x, ids, w, W13_mx, W2_mx, bufs.expert_offsets, bufs.perm, bufs.out, bufs.ws,
                      d_num_tokens=d_T)
        torch.cuda.synchronize()
        assert B.moe_last_device_error(bufs.ws) & B.MOE_DEVERR_BAD_EXPERT_ID
        B.moe_clear_device_error(bufs.ws)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                B.moe_forward(p, x, ids, w, W13_mx, W2_mx, bufs.expert_offsets, bufs.perm, bufs.out, bufs.ws,
                              d_num_tokens=d_T, stream=s)
        torch.cuda.current_stream().wait_stream(s)
        for T_dev in (12, 5, 1, 0):
            d_T.fill_(T_dev)
            bufs.out.fill_(4.0)
            g.replay()
            torch.cuda.synchronize()
            assert torch.all(bufs.out[T_dev:] == 4.0)
            valid = int(np.count_nonzero((ids_np[:T_dev] >= 0) & (ids_np[:T_dev] < E)))
            assert int(bufs.expert_offsets[-1]) == valid
            if T_dev == 0:
                continue
            eager = B.Buffers(p)
            B.moe_forward(p, x, ids, w, W13_mx, W2_mx, eager.expert_offsets, eager.perm, eager.out, eager.ws,
                          d_num_tokens=d_T)
            torch.cuda.synchronize()
            assert torch.equal(bufs.out[:T_dev].view(torch.int16), eager.out[:T_dev].view(torch.int16))
            ref_acc, _, bad = oracle.moe_tokens(wlm.bf16_bits(x), ids_np, w_np, W13_d, W2_d,
                                                tokens=np.arange(T_dev, dtype=np.int32))
            assert_within_tolerance(wlm.bf16_bits(bufs.out[:T_dev]), ref_acc, f"mxfp8 edge form {form} T={T_dev}")
