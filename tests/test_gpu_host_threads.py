"""Host threads calling moe_forward at the same time, each on its own stream
with its own workspace and buffers, get the bits of the same calls made one
at a time: the library keeps its launch caches (kernel attributes set, the
device checked, the SM count) per host thread, and everything a call keeps
on the GPU lives in its own workspace. One case per GEMM placement: CTA
pairs, single-CTA tiles, the fused decode kernel (a cooperative launch) and
its one-kernel form."""
from __future__ import annotations

import threading

import pytest
import torch

import workloads as wlm
from parity import DeviceWorkload

pytestmark = pytest.mark.gpu

# (T, E, k, H, I), path, forward form
CASES = [((1024, 8, 2, 512, 256), 1, 0), ((256, 16, 4, 512, 256), 3, 0), ((8, 64, 4, 512, 256), 2, 1),
         ((8, 64, 4, 512, 256), 2, 2)]


@pytest.fixture(scope="module")
def B():
    from moe_routed_expert_routing_gb300.build import build
    build()
    from moe_routed_expert_routing_gb300 import binding
    return binding


def test_concurrent_host_threads_match_calls_made_alone(B):
    runs = []
    for i, (shape, path, form) in enumerate(CASES):
        wl = wlm.custom("threads", *shape, seed=60 + i)
        dw = DeviceWorkload(wl)
        p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, path=path, forward_form=form)
        alone = B.Buffers(p)
        B.moe_forward(p, dw.x, dw.ids, dw.w, dw.W13, dw.W2, alone.expert_offsets, alone.perm, alone.out, alone.ws)
        torch.cuda.synchronize()
        assert B.moe_last_device_error(alone.ws) == 0
        runs.append((p, dw, alone.out.clone(), B.Buffers(p), torch.cuda.Stream()))
    torch.cuda.synchronize()

    failures = []
    start = threading.Barrier(len(runs))

    def work(i):
        p, dw, ref, bufs, s = runs[i]
        try:
            start.wait()
            for _ in range(5):
                B.moe_forward(p, dw.x, dw.ids, dw.w, dw.W13, dw.W2, bufs.expert_offsets, bufs.perm, bufs.out,
                              bufs.ws, stream=s)
            s.synchronize()
            if B.moe_last_device_error(bufs.ws) != 0:
                failures.append((i, "device error"))
            elif not torch.equal(bufs.out.view(torch.int16), ref.view(torch.int16)):
                failures.append((i, "bits differ"))
        except Exception as e:   # reported below, on the main thread
            failures.append((i, repr(e)))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(runs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads)
    assert not failures, failures
