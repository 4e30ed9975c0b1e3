"""Host logic of the co-resident launch (CPU only, no GPU): the kernels whose
CTAs wait on one another (the fused decode kernel in both forms) are sized
against the occupancy the device reports and launched cooperatively; when
not even one CTA fits on an SM the launch is refused before it is made,
instead of starting a grid whose waits could only run out.

The decision is `moe::coresident_grid` in csrc/moe_internal.h; this test
compiles a small host program against that header with nvcc and runs it.
"""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "moe_routed_expert_routing_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "moe_internal.h"
int main()
{
    struct Case { long long want; int per_sm, sms, grid; };
    const Case cases[] = {
        {152, 1, 152, 152},   // one CTA per SM on every SM: the whole grid
        {144, 1, 152, 144},   // fewer units than SMs: one CTA per unit
        {400, 1, 152, 152},   // more units than fit: capped at what is resident at once
        {400, 2, 152, 304},
        {152, 0, 152, 0},     // the kernel fits on no SM: refused
        {0, 1, 152, 0},       // nothing to launch
        {152, 1, 0, 0},       // no SM count
    };
    int bad = 0;
    for (const Case &c : cases) {
        const int g = moe::coresident_grid(c.want, c.per_sm, c.sms);
        if (g != c.grid) {
            std::printf("want=%lld per_sm=%d sms=%d: grid %d, expected %d\n", c.want, c.per_sm, c.sms, g, c.grid);
            ++bad;
        }
    }
    std::printf(bad ? "FAIL\n" : "OK\n");
    return bad;
}
"""


def test_coresident_grid_refuses_and_caps(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    src = tmp_path / "coresident.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "coresident"
    r = subprocess.run([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-I", CSRC,
                        "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "OK", r.stdout + r.stderr
