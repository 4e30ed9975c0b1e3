"""Failure detection without a GPU fault: a bounded wait that runs out.

The fused decode kernel's down units wait, with a time limit, until every
gate-up unit of their expert has counted itself in a per-expert readiness
count in the workspace header. Setting those counts to a value the gate-up
units cannot bring to the target makes every such wait run out (nothing ever
satisfies it). The kernel then stops its pipelines in order (in-flight TMA
loads and MMAs drained, TMEM freed), sets MOE_DEVERR_WAIT_TIMEOUT in the
device error word, and its last CTA still returns the counters to zero, so
that after moe_clear_device_error the same workspace gives the same bits as
before. The limit is 2 s, so each case takes a few seconds."""
from __future__ import annotations

import time

import pytest
import torch

import workloads as wlm
from parity import DeviceWorkload

pytestmark = pytest.mark.gpu

HEADER_BYTES = 256 + 4 * (1024 + 2)   # error word block, readiness counts, done, exits


@pytest.fixture(scope="module")
def B():
    from moe_routed_expert_routing_gb300.build import build
    build()
    from moe_routed_expert_routing_gb300 import binding
    return binding


def _forward(B, p, dw, bufs, W13, W2):
    B.moe_forward(p, dw.x, dw.ids, dw.w, W13, W2, bufs.expert_offsets, bufs.perm, bufs.out, bufs.ws)
    torch.cuda.synchronize()


@pytest.mark.parametrize("form,layout", [(1, 0), (2, 0), (1, 2)], ids=["separate", "one_kernel", "separate_mxfp8"])
def test_wait_limit_reports_and_recovers(B, form, layout):
    wl = wlm.custom("timeout", 8, 64, 4, 512, 256, seed=71)
    dw = DeviceWorkload(wl)
    p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, forward_form=form, weight_layout=layout)
    assert B.moe_resolve_profile(p)["fused_mlp"] == 1
    W13, W2 = (B.moe_quantize_weights(p, dw.W13, dw.W2) if layout == B.MOE_WEIGHTS_MXFP8 else (dw.W13, dw.W2))
    bufs = B.Buffers(p)
    _forward(B, p, dw, bufs, W13, W2)
    assert B.moe_last_device_error(bufs.ws) == 0
    clean = bufs.out.clone()

    # readiness counts far below zero: no down unit's wait can be satisfied
    ready = bufs.ws[256:256 + 4 * wl.E].view(torch.int32)
    ready.fill_(-(1 << 30))
    t0 = time.time()
    _forward(B, p, dw, bufs, W13, W2)
    took = time.time() - t0
    err = B.moe_last_device_error(bufs.ws)
    assert err & B.MOE_DEVERR_WAIT_TIMEOUT, err
    assert 1.5 < took < 60.0, took                                  # the 2 s limit ran out, once per wait chain
    assert int(bufs.ws[4:HEADER_BYTES].count_nonzero()) == 0      # tail clean-up zeroed every counter

    B.moe_clear_device_error(bufs.ws)
    _forward(B, p, dw, bufs, W13, W2)
    assert B.moe_last_device_error(bufs.ws) == 0
    assert torch.equal(bufs.out.view(torch.int16), clean.view(torch.int16))
