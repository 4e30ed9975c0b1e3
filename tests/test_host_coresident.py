"""Host logic of the co-resident launch (CPU only, no GPU): the kernels whose
CTAs wait on one another (the fused decode kernel in both forms) are sized
against the occupancy the device reports and launched cooperatively; when
not even one CTA fits on an SM the launch is refused before it is made,
instead of starting a grid whose waits could only run out.

The decision is `moe::coresident_grid` in csrc/moe_internal.h, with
`moe::fused_grid_sms` (the fused decode kernel leaves one SM to the dispatch
block where its gate-up units fit one wave on one SM fewer); this test
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
    // the fused decode kernel's grid: one SM left to the dispatch where the
    // gate-up units (row tiles bound x ceil(I / 128)) fit one wave on one SM fewer
    struct Fused { bool mega, fp8; long long cap; int E, I, tile_rows, sms, grid_sms; };
    const Fused fused[] = {
        {false, false, 6, 384, 3072, 16, 152, 151},      // one token, k=6: 6 row tiles x 24 = 144 units
        {false, false, 48, 384, 3072, 16, 152, 152},     // eight tokens: (48 + 3) x 24 units
        {true, false, 6, 384, 3072, 16, 152, 152},       // one-kernel form: no dispatch kernel before it
        {false, true, 6, 384, 3072, 16, 152, 152},       // MXFP8 weights: the full grid
        {false, false, 8, 384, 2304, 16, 152, 151},      // 8 x 18 = 144 units
        {false, false, 8, 384, 2432, 16, 152, 152},      // 8 x 19 = 152 units: more than 151
        {false, false, 6, 4, 3072, 16, 152, 151},        // more slots than experts: min(cap, E) row tiles
        {false, false, 6, 384, 3072, 16, 1, 1},          // a single SM keeps it
    };
    for (const Fused &f : fused) {
        const int g = moe::fused_grid_sms(f.mega, f.fp8, f.cap, f.E, f.I, f.tile_rows, f.sms);
        if (g != f.grid_sms) {
            std::printf("fused mega=%d fp8=%d cap=%lld E=%d I=%d sms=%d: %d SMs, expected %d\n", f.mega, f.fp8,
                        f.cap, f.E, f.I, f.sms, g, f.grid_sms);
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
