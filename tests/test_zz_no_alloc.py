"""moe_dispatch_noalloc: the dispatch entry point for callers that cannot
allocate device memory (a runtime whose device memory is fixed at start-up,
or code under stream capture, where cudaMalloc is illegal). It keeps its
scratch in a static device array inside libmoe.so instead of a caller
workspace. Its results must equal moe_dispatch's, call after call, since all
calls share that one array, and the oracle's dispatch bit for bit. Collected
last so that a failure here does not stop the rest of a run early; it also
passes alone in a fresh process.
"""
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


def _outputs(p, device="cuda"):
    return (torch.full((p.E + 1,), -7, dtype=torch.int32, device=device),
            torch.full((p.cap,), -7, dtype=torch.int32, device=device),
            torch.full((p.T_max * p.k,), -7, dtype=torch.int32, device=device),
            torch.zeros((p.cap, p.H), dtype=torch.bfloat16, device=device))


def _same(a, b, n_rows):
    offs_a, perm_a, inv_a, xs_a = a
    offs_b, perm_b, inv_b, xs_b = b
    assert torch.equal(offs_a, offs_b)
    assert torch.equal(perm_a[:n_rows], perm_b[:n_rows])
    assert torch.equal(inv_a, inv_b)
    assert torch.equal(xs_a[:n_rows].view(torch.int16), xs_b[:n_rows].view(torch.int16))


def test_noalloc_dispatch_matches_workspace_dispatch_two_calls_in_a_row(B):
    # two different problems back to back: the second reuses the static array
    # the first one left behind
    for name, seed in [("large", None), ("small", 5)]:
        wl = wlm.WORKLOADS[name]
        ids_np, _ = wlm.make_routing(wl, seed)
        if name == "small":
            ids_np[3, 1] = -1                      # a dropped slot
        ids = torch.from_numpy(ids_np).cuda()
        x = wlm.make_x(wl, "cuda")
        p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I)

        ref = _outputs(p)
        ws = torch.zeros(B.moe_workspace_size(p), dtype=torch.uint8, device="cuda")
        B.moe_dispatch(p, ids, ref[0], ref[1], ref[2], ws, x=x, x_sorted=ref[3])

        got = _outputs(p)
        B.moe_dispatch_noalloc(p, ids, got[0], got[1], got[2], x=x, x_sorted=got[3])
        torch.cuda.synchronize()
        n_rows = int(ref[0][-1].item())
        assert n_rows == int(np.count_nonzero(ids_np >= 0))
        _same(got, ref, n_rows)


def test_noalloc_dispatch_repeated_with_device_token_count(B):
    wl = wlm.custom("na", 300, 24, 4, 256, 128, seed=12)
    ids_np, _ = wlm.make_routing(wl)
    ids = torch.from_numpy(ids_np).cuda()
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I)
    ws = torch.zeros(B.moe_workspace_size(p), dtype=torch.uint8, device="cuda")
    for T_dev in (300, 17):
        d_T = torch.tensor([T_dev], dtype=torch.int32, device="cuda")
        ref = _outputs(p)
        got = _outputs(p)
        B.moe_dispatch(p, ids, ref[0], ref[1], ref[2], ws, d_num_tokens=d_T)
        B.moe_dispatch_noalloc(p, ids, got[0], got[1], got[2], d_num_tokens=d_T)
        torch.cuda.synchronize()
        _same(got[:3] + (ref[3],), ref, int(ref[0][-1].item()))


def test_noalloc_dispatch_rejects_problems_beyond_its_static_scratch(B):
    # 64 + 2 * ceil(T*k / 1024) * E ints must fit in MOE_NOALLOC_SCRATCH_INTS
    p = B.Problem.make(65536, 1024, 8, 256, 128)
    fake = 1 << 40    # never dereferenced: the size check comes first
    with pytest.raises(B.MoeError) as ei:
        B.moe_dispatch_noalloc(p, fake, fake, fake, fake)
    assert ei.value.status == 4


def test_noalloc_dispatch_matches_oracle(B):
    """Bit-exact against the oracle's stable dispatch on its own, at the
    prefill shape (12 dispatch blocks), with a dropped slot and experts 0..4
    given 1000 more slots each across two blocks (slot 5 of those tokens may
    repeat one of them: duplicates are two rows, as in the oracle)."""
    wl = wlm.WORKLOADS["prefill"]
    ids_np, _ = wlm.make_routing(wl)
    ids_np[7, 2] = -1
    ids_np[100:1100, :5] = np.arange(5, dtype=np.int32)   # experts 0..4 each hold 1000 more slots in a row
    ids = torch.from_numpy(ids_np).cuda()
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I)
    for _ in range(2):
        got = _outputs(p)
        B.moe_dispatch_noalloc(p, ids, got[0], got[1], got[2])
        torch.cuda.synchronize()
        _, o_off, o_perm, o_inv, n_bad = oracle.dispatch(ids_np, wl.E)
        n_rows = int(o_off[-1])
        assert n_bad == 0 and n_rows == wl.R - 1
        assert np.array_equal(got[0].cpu().numpy(), o_off)
        assert np.array_equal(got[1].cpu().numpy()[:n_rows], o_perm[:n_rows])
        assert np.array_equal(got[2].cpu().numpy(), o_inv)
