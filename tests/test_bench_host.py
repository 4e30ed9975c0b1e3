"""Host-side logic of bench.py on CPU: the replica aggregation over ranks
(world size 2, gloo), FLOP/byte accounting, and the reference arm's line."""
from __future__ import annotations

import json
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
import workloads as wlm


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    bench.init_dist(world, rank, backend="gloo")
    local_ms = 10.0 + 5.0 * rank
    mx = bench.max_over_ranks(local_ms, world)
    sm = bench.sum_over_ranks(1.0, world)
    bench.barrier(world)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((rank, mx, sm))


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 15.0, 2.0), (1, 15.0, 2.0)]


def test_single_rank_aggregation_is_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.sum_over_ranks(2.0, 1) == 2.0


def test_call_accounting():
    wl = wlm.custom("acc", 4, 8, 2, 256, 128)
    ids = np.array([[0, 1], [1, 2], [2, 3], [3, -1]], dtype=np.int32)
    a = bench.call_accounting(wl, ids)
    assert a["R"] == 7 and a["touched_experts"] == 4
    assert a["flops"] == 6 * 7 * 256 * 128
    assert a["gemm1_flops"] == 4 * 7 * 256 * 128
    assert a["bytes"] == 4 * 6 * 256 * 128 + 2 * 4 * 256 * 2 + 8 * 7
    assert a["gemm1_bytes"] == 4 * 4 * 128 * 256 + 2 * 7 * 256 + 2 * 7 * 128
    # MXFP8 weights: one code byte per element plus one scale byte per 32
    m = bench.call_accounting(wl, ids, weight_bytes=33 / 32)
    assert m["bytes"] == 4 * 3 * (33 / 32) * 256 * 128 + 2 * 4 * 256 * 2 + 8 * 7
    assert m["flops"] == a["flops"]


def test_defaults():
    a = bench.parse_args([])
    # the headline is the largest single-GPU configuration (T=8192, E=128, k=8, H=4096, I=1536)
    assert a.gpus == 1 and a.impl == "ours" and a.workload == "large" and a.warmup >= 3
    assert a.per_config


def test_reference_arm_line_on_tiny(capsys, monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    assert bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1


def test_reference_arm_other_ranks_exit_quietly(capsys, monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    assert bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out.strip() == ""


def test_traffic_key_ignores_comments_not_code():
    """The ncu traffic captures stay keyed to the kernel code: comments and
    layout do not change the key, a changed token does."""
    src = "int a = 1; // note\n/* block\n comment */  int b =  2;\n"
    assert bench.code_only(src) == bench.code_only("int a = 1;\n   int b = 2; // other note\n")
    assert bench.code_only(src) != bench.code_only("int a = 1; int b = 3;")
    assert bench.kernel_sha() == bench.kernel_sha()


def test_traffic_key_selection():
    """Each workload's dominant kernel maps to its own capture."""
    def inp(path):
        return {"path": (path, 128)}
    assert bench.traffic_key([inp(2), inp(2)], "bf16", True) == "fused_small"
    assert bench.traffic_key([inp(2)], "mxfp8", True) == "fused_small_mxfp8"
    assert bench.traffic_key([inp(2)], "bf16", False) == "gate_up_small_m"
    assert bench.traffic_key([inp(3)], "bf16", False) == "gate_up_tiled"
    assert bench.traffic_key([inp(1)], "bf16", False) == "gate_up_pair"
    assert bench.traffic_key([inp(1), inp(3)], "bf16", False) is None
    for key in ("fused_small", "fused_small_mxfp8", "gate_up_small_m", "gate_up_tiled", "gate_up_pair"):
        cap = bench.NCU_TRAFFIC[key]
        assert cap["traffic"] > 0 and 0.9 < cap["traffic"] / cap["algorithmic"] < 1.3


@pytest.mark.gpu
def test_gpu_arm_json_line_on_tiny(capsys, monkeypatch):
    """The GPU arm's one JSON line carries every key of the measurement
    contract (tiny workload, a few steps)."""
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    assert bench.main(["--workload", "tiny", "--steps", "20", "--warmup", "3", "--e2e-steps", "5",
                       "--cpu-seconds", "0.5", "--no-per-config"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                "gpu_launches", "clocks"):
        assert key in line, key
    assert line["value"] > 0 and line["n_gpus"] == 1 and line["gpu_launches"] > 0
    r = line["roofline"]
    assert r["bound"] in ("hbm", "tensor") and r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    assert line["e2e"]["h2d_bytes_per_step"] > 0 and line["e2e"]["d2h_bytes_per_step"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(line["clocks"])
    # warm-up is honoured exactly, and the dominant kernel's time per step
    # cannot exceed the step
    assert line["warmup"] == 3 and line["steps"] == 20
    assert r["kernel_us_per_launch"] * len(line["config"]["batches_per_step"]) <= line["ms_per_step"] * 1e3 + 1e-6
    assert r["algorithmic_per_launch"] / (r["kernel_us_per_launch"] * 1e-6) / (1e12 if r["unit"] == "TFLOP/s"
                                                                             else 1e9) == pytest.approx(r["achieved"])


@pytest.mark.gpu
def test_gpu_arm_per_config_block(capsys, monkeypatch):
    """The per-config block times prefill, the Zipf small batch and decode on
    their own (shrunk here to E=8, T=16 so that the test is quick)."""
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    assert bench.main(["--workload", "tiny", "--steps", "5", "--warmup", "3", "--e2e-steps", "2",
                       "--no-cpu-baseline", "--experts", "8", "--tokens", "16", "--config-ms", "5"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    pc = line["per_config"]
    for name in ("prefill", "small", "decode"):
        e = pc[name]
        assert e["ms_per_step"] > 0 and e["tflops"] > 0 and 0 < e["call_roofline"]["frac"]
        assert e["dominant_kernel"]["kernel_us_per_launch"] <= e["ms_per_step"] * 1e3 + 1e-6
    # decode's two batches are also timed each in a graph of its own
    alone = pc["decode"]["us_per_call_alone"]
    assert set(alone) == set(pc["decode"]["us_per_call"]) and len(alone) == 2
    assert all(v > 0 for v in alone.values())
    assert pc["prefill"]["us_per_call_alone"] == {}


def test_clock_samples_restricted_to_the_timed_region():
    """Only nvidia-smi samples whose timestamps fall inside the timed region
    count; with none inside, all of them count and the line says so."""
    import datetime
    t0 = datetime.datetime(2026, 12, 3, 6, 0, 0)

    def line(ms, mhz, watts, cap="Not Active"):
        ts = (t0 + datetime.timedelta(milliseconds=ms)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return f"{ts}, 0, {mhz}, 2070, {watts}, 0x0, Not Active, Not Active, Not Active, {cap}\n"

    lines = [line(0, 2070, 150), line(100, 1800, 1390, "Active"), line(110, 1820, 1395, "Active"), line(300, 2070, 200)]
    base = t0.timestamp()
    inside = bench.ClockSampler.parse(lines, (base + 0.05, base + 0.2))
    assert inside["samples"] == 2 and inside["sm_mhz"] == 1810.0 and inside["reasons"] == ["sw_power_cap"]
    assert inside["power_w_max"] == 1395.0 and inside["samples_from"] == "the timed region"
    none_inside = bench.ClockSampler.parse(lines, (base + 0.5, base + 0.6))
    assert none_inside["samples"] == 4 and none_inside["samples_from"].startswith("around")
    assert bench.ClockSampler.parse(lines)["samples_from"] == "the whole sampling run"
    assert bench.ClockSampler.parse(["garbage\n"]) is None
