"""GPU parity: dispatch (bit-exact indices and offsets) and combine (bit-exact
given the same sorted batch), through the C ABI, against the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as wlm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from moe_routed_expert_routing_gb300.build import build
    build()
    from moe_routed_expert_routing_gb300 import binding
    return binding


def run_dispatch(B, p, ids_t, x=None, d_T=None):
    offs = torch.full((p.E + 1,), -7, dtype=torch.int32, device="cuda")
    perm = torch.full((p.cap,), -7, dtype=torch.int32, device="cuda")
    inv = torch.full((p.T_max * p.k,), -7, dtype=torch.int32, device="cuda")
    ws = torch.zeros(B.moe_workspace_size(p), dtype=torch.uint8, device="cuda")
    xs = None
    if x is not None:
        xs = torch.zeros((p.cap, p.H), dtype=torch.bfloat16, device="cuda")
    B.moe_dispatch(p, ids_t, offs, perm, inv, ws, x=x, x_sorted=xs, d_num_tokens=d_T)
    torch.cuda.synchronize()
    return offs.cpu().numpy(), perm.cpu().numpy(), inv.cpu().numpy(), xs, ws


def check_dispatch_exact(ids_np, E, offs, perm, inv, T=None):
    T = ids_np.shape[0] if T is None else T
    counts, o_off, o_perm, o_inv, _ = oracle.dispatch(ids_np[:T], E)
    n = int(o_off[-1])
    assert np.array_equal(offs, o_off)
    assert np.array_equal(perm[:n], o_perm[:n])
    assert np.array_equal(inv[:T * ids_np.shape[1]], o_inv)


@pytest.mark.parametrize("name", ["tiny", "decode1", "decode8", "small", "prefill", "large"])
def test_dispatch_bit_exact(B, name):
    wl = wlm.WORKLOADS[name]
    ids_np, _ = wlm.make_routing(wl)
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I)
    x = wlm.make_x(wl, "cuda")
    offs, perm, inv, xs, ws = run_dispatch(B, p, torch.from_numpy(ids_np).cuda(), x=x)
    check_dispatch_exact(ids_np, wl.E, offs, perm, inv)
    n = int(offs[-1])
    assert n == wl.R
    # gather: x_sorted[row] == x[perm[row] // k], byte for byte
    src = torch.from_numpy(perm[:n] // wl.k).long().cuda()
    assert torch.equal(xs[:n].view(torch.int16), x[src].view(torch.int16))
    assert B.moe_last_device_error(ws) == 0


@pytest.mark.parametrize("T_dev", [0, 1, 37, 64])
def test_dispatch_dynamic_token_count(B, T_dev):
    wl = wlm.custom("dyn", 64, 16, 4, 256, 128, seed=3)
    ids_np, _ = wlm.make_routing(wl)
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I)
    d_T = torch.tensor([T_dev], dtype=torch.int32, device="cuda")
    offs, perm, inv, _, _ = run_dispatch(B, p, torch.from_numpy(ids_np).cuda(), d_T=d_T)
    check_dispatch_exact(ids_np, wl.E, offs, perm, inv, T=T_dev)


@pytest.mark.parametrize("T", [300, 900])   # one dispatch block / three blocks
def test_dispatch_dropped_and_invalid_ids(B, T):
    rng = np.random.default_rng(4)
    k, E = 3, 10
    ids_np = rng.integers(0, E, (T, k)).astype(np.int32)
    ids_np[5, 1] = -1
    ids_np[17, 0] = -1
    ids_np[40, 2] = E + 3          # invalid: dropped and flagged
    p = B.Problem.make(T, E, k, 256, 128)
    offs, perm, inv, _, ws = run_dispatch(B, p, torch.from_numpy(ids_np).cuda())
    check_dispatch_exact(ids_np, E, offs, perm, inv)
    assert offs[-1] == T * k - 3
    assert B.moe_last_device_error(ws) & B.MOE_DEVERR_BAD_EXPERT_ID
    B.moe_clear_device_error(ws)
    assert B.moe_last_device_error(ws) == 0


@pytest.mark.parametrize("T,k,E", [(3000, 4, 1000), (2500, 8, 48), (4096, 2, 33), (1100, 1, 1), (9000, 8, 700)])
def test_dispatch_many_blocks_any_expert_count(B, T, k, E):
    """Multi-block dispatch (count, scan, scatter) at expert counts from 1 to
    1000, powers of two or not, against the oracle, bit-exact."""
    rng = np.random.default_rng(T + E)
    ids_np = np.stack([rng.choice(E, size=k, replace=False) if E >= k else rng.integers(0, E, size=k)
                       for _ in range(T)]).astype(np.int32)
    p = B.Problem.make(T, E, k, 256, 128)
    offs, perm, inv, _, ws = run_dispatch(B, p, torch.from_numpy(ids_np).cuda())
    check_dispatch_exact(ids_np, E, offs, perm, inv)
    assert int(offs[-1]) == T * k and B.moe_last_device_error(ws) == 0


def test_dispatch_one_hot_expert_many_blocks(B):
    # 5000 slots all on expert 2: spans several dispatch blocks; stability = identity order
    T, k, E = 5000, 1, 4
    ids_np = np.full((T, k), 2, dtype=np.int32)
    p = B.Problem.make(T, E, k, 256, 128)
    offs, perm, inv, _, _ = run_dispatch(B, p, torch.from_numpy(ids_np).cuda())
    assert offs.tolist() == [0, 0, 0, T, T]
    assert np.array_equal(perm[:T], np.arange(T))
    check_dispatch_exact(ids_np, E, offs, perm, inv)


@pytest.mark.parametrize("shape", [(64, 8, 2, 256), (1, 384, 6, 7168), (300, 24, 8, 512), (2048, 384, 6, 1024)])
def test_combine_bit_exact(B, shape):
    T, E, k, H = shape
    wl = wlm.custom("c", T, E, k, H, 128, seed=T + E)
    ids_np, w_np = wlm.make_routing(wl)
    ids_np[0, -1] = -1 if T > 1 else ids_np[0, -1]
    p = B.Problem.make(T, E, k, H, 128)
    offs, perm, inv, _, _ = run_dispatch(B, p, torch.from_numpy(ids_np).cuda())
    n = int(offs[-1])
    g = torch.Generator(device="cuda").manual_seed(9)
    y_sorted = torch.randn((p.cap, H), generator=g, device="cuda")
    out = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    inv_t = torch.from_numpy(inv).cuda()
    w_t = torch.from_numpy(w_np).cuda()
    B.moe_combine(p, y_sorted, inv_t, w_t, out)
    torch.cuda.synchronize()
    ref_acc, ref = oracle.combine_sorted(y_sorted[:max(n, 1)].cpu().numpy(), inv, w_np)
    assert np.array_equal(wlm.bf16_bits(out), ref)


def test_identity_expert_dispatch_then_combine(B):
    """Dispatch + combine with y_sorted = x_sorted reproduces sum_j w * x (closed form)."""
    wl = wlm.custom("id", 200, 16, 4, 512, 128, seed=5)
    ids_np, w_np = wlm.make_routing(wl)
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I)
    x = wlm.make_x(wl, "cuda")
    offs, perm, inv, xs, _ = run_dispatch(B, p, torch.from_numpy(ids_np).cuda(), x=x)
    out = torch.zeros_like(x)
    B.moe_combine(p, xs.float(), torch.from_numpy(inv).cuda(), torch.from_numpy(w_np).cuda(), out)
    torch.cuda.synchronize()
    ref = (w_np.astype(np.float64).sum(1)[:, None]) * x.double().cpu().numpy()
    got = out.double().cpu().numpy()
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-6)


def test_combine_dynamic_token_count_leaves_tail(B):
    T, E, k, H = 50, 8, 2, 256
    wl = wlm.custom("cd", T, E, k, H, 128, seed=6)
    ids_np, w_np = wlm.make_routing(wl)
    p = B.Problem.make(T, E, k, H, 128)
    d_T = torch.tensor([20], dtype=torch.int32, device="cuda")
    offs, perm, inv, _, _ = run_dispatch(B, p, torch.from_numpy(ids_np).cuda(), d_T=d_T)
    y_sorted = torch.randn((p.cap, H), device="cuda")
    out = torch.full((T, H), 3.0, dtype=torch.bfloat16, device="cuda")
    B.moe_combine(p, y_sorted, torch.from_numpy(inv).cuda(), torch.from_numpy(w_np).cuda(), out, d_num_tokens=d_T)
    torch.cuda.synchronize()
    _, ref = oracle.combine_sorted(y_sorted.cpu().numpy(), inv[:20 * k], w_np[:20])
    assert np.array_equal(wlm.bf16_bits(out[:20]), ref)
    assert torch.all(out[20:] == 3.0)
