#!/usr/bin/env python
"""Benchmark of routed-MoE expert execution on one GB300 (or N replicas).

One step = one pass of the whole path (dispatch -> gate-up GEMM with fused
SiLU*up -> down GEMM -> combine) over each batch of the chosen workload. The
default workload is the largest single-GPU configuration: T=8192 tokens,
E=128 experts, top-8, H=4096, I=1536, a quarter of the tokens forced onto
expert 0 (the tensor-bound case). Weights, routing and activations are
synthetic (seeded generators in workloads.py) and resident in HBM.

Timing: one step is captured in a CUDA graph. Warm-up is exactly W steps
(one eager forward, which also sets the kernels' function attributes, then
W-1 replays); then exactly K replays between two CUDA events, barrier +
synchronize on both sides, max over ranks. The touched expert weights and
sorted batches of one step (~5.5 GB for the default workload) are far larger
than the 129 MB L2, so no flush is needed between steps.

Printed: one JSON line (rank 0) with the throughput (TFLOP/s), the roofline
of the dominant kernel (its share of a profiled step, from CUDA events
between the stages, applied to the timed step), an end-to-end number through
the public C-ABI call with pinned host buffers, SM clocks sampled during the
timed region, the CPU oracle's throughput on a bounded sample, and, under
`per_config`, us/call, TFLOP/s and call-roofline fraction of the prefill,
Zipf small-batch and decode workloads, each timed on its own.

``--impl reference`` times the CPU oracle instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wlm  # noqa: E402

WORKLOAD_SETS = {
    "decode": ["decode1", "decode8"],
    "tiny": ["tiny"],
    "decode1": ["decode1"],
    "decode8": ["decode8"],
    "small": ["small"],
    "prefill": ["prefill"],
    "large": ["large"],
}
STAGES = ["dispatch", "gather", "gemm_gate_up", "gemm_down", "combine"]
GRAPH_STEPS = 10

# DRAM traffic of the dominant kernel (dram__bytes_read.sum + dram__bytes_write.sum
# per launch) from ncu captures of small cases of each workload that keep its
# per-expert shape and rows per expert, with that kernel's algorithmic bytes per
# launch in the same case (the `roofline.algorithmic_bytes_per_launch` of the
# captured command's own bench line). A full launch's traffic is the captured
# ratio times its own algorithmic bytes: the units (touched experts, row tiles)
# grow and the bytes with them. Keyed to the sha256 of the GEMM sources at
# capture time, comments and layout left out: after any change to the code,
# traffic reports null.
NCU_TRAFFIC = {
    "kernel_sha256": "7cbba4c501754ca48fbfdb6f5bb374f95efe5c08adc202f542e4a2fd3bd61c9a",
    "fused_small": {"case": "decode T=8 shape with E=24", "traffic": 2.644598e+09, "algorithmic": 2.644378e+09},
    "fused_small_mxfp8": {"case": "decode T=8 shape with E=24, MXFP8 weights", "traffic": 1.364904e+09, "algorithmic": 1.364460e+09},
    "gate_up_small_m": {"case": "Zipf small batch with E=128", "traffic": 6.938921e+09, "algorithmic": 6.947865e+09},
    "gate_up_tiled": {"case": "prefill shape with T=256, E=48", "traffic": 4.260334e+09, "algorithmic": 4.259316e+09},
    "gate_up_pair": {"case": "large shape with T=4096, E=64", "traffic": 1.984390e+09, "algorithmic": 1.979711e+09},
}


# ----------------------------------------------------------------------------- accounting

def call_accounting(wl: wlm.Workload, ids_np: np.ndarray, weight_bytes: float = 2.0) -> dict:
    """FLOPs and algorithmic bytes of one forward over this routing;
    weight_bytes per weight element: 2 (bf16), 33/32 (MXFP8 codes + scales)."""
    R = int(np.count_nonzero(ids_np >= 0))
    touched = int(np.unique(ids_np[ids_np >= 0]).size)
    T, H, I = wl.T, wl.H, wl.I
    wb = weight_bytes
    return {
        "flops": 6.0 * R * H * I,
        "bytes": touched * 3.0 * wb * H * I + 2.0 * T * H * 2 + 8.0 * R,
        "gemm1_flops": 4.0 * R * H * I,
        "gemm1_bytes": touched * 2.0 * wb * I * H + 2.0 * R * H + 2.0 * R * I,
        "gemm2_bytes": touched * wb * H * I + 2.0 * R * I + 2.0 * R * H,
        "touched_experts": touched,
        "R": R,
    }


def traffic_key(inputs, weights: str, fused: bool):
    """Which captured kernel the dominant kernel of these inputs is."""
    if fused:
        return "fused_small_mxfp8" if weights == "mxfp8" else "fused_small"
    paths = {d["path"][0] for d in inputs}
    return {frozenset({2}): "gate_up_small_m", frozenset({3}): "gate_up_tiled",
            frozenset({1}): "gate_up_pair"}.get(frozenset(paths))


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def code_only(text: str) -> str:
    """C++ source without comments and with whitespace collapsed: edits to
    comments or layout leave the kernels, and so their captures, unchanged."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_sha() -> str:
    h = hashlib.sha256()
    for name in ("grouped_gemm.cu", "ptx.cuh", "moe_internal.h"):
        with open(os.path.join(ROOT, "moe_routed_expert_routing_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()


# ----------------------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, local: int, backend: str = "nccl"):
    if world <= 1:
        return
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    if backend == "nccl":
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        dist.init_process_group(backend)


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return float(value)
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return float(value)
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock, power and throttle reasons, every 10 ms,
    each with its timestamp; stop() keeps the samples that fall inside the
    window marked by mark_start() / mark_end() (the timed region), or all of
    them, with a note, if none does."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.window = None
        self.path = os.path.join("/tmp", f"moe_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "10"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def mark_start(self):
        self._t0 = time.time()

    def mark_end(self):
        self.window = (self._t0, time.time())

    @staticmethod
    def parse(lines, window=None):
        """Samples of nvidia-smi's csv lines (see QUERY), restricted to `window`
        (two epoch seconds) when given; returns the summary dict or None."""
        import datetime
        rows = []
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), float(parts[4]), parts[6:10]))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if window and window[0] <= r[0] <= window[1]]
        use = inside or rows
        reasons = sorted({n for r in use for n, v in zip(ClockSampler.REASONS, r[4]) if v.lower().startswith("active")})
        out = {"sm_mhz": float(np.median([r[1] for r in use])), "sm_max_mhz": float(max(r[2] for r in use)),
               "reasons": reasons, "samples": len(use), "power_w_max": float(max(r[3] for r in use))}
        out["samples_from"] = ("the whole sampling run" if not window else "the timed region" if inside else
                               "around the timed region (no sample fell inside it)")
        return out

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        return self.parse(lines, self.window)


# ----------------------------------------------------------------------------- CPU oracle

def time_oracle(inputs, seconds: float, tokens_cap: int | None = None, host_cache: dict | None = None) -> dict:
    """The oracle, as it stands, on the host cores over a bounded sample.
    host_cache (optional) keeps the host copies of the sampled experts'
    weights between calls on the same sample; only the oracle calls are timed."""
    import oracle
    oracle.load()
    cores = len(os.sched_getaffinity(0))
    flops_done, t_total, runs = 0.0, 0.0, 0
    samples = []
    for d in inputs:
        wl = d["wl"]
        T = wl.T
        n_tok = T if tokens_cap is None else max(1, min(T, tokens_cap))
        key = (id(d), n_tok)
        if host_cache is not None and key in host_cache:
            samples.append(dict(host_cache[key]))
            continue
        tok = np.arange(n_tok, dtype=np.int32) if n_tok == T else wlm.token_subset(wl, n_tok)
        ids = d["ids_np"]
        touched = np.unique(ids[tok][ids[tok] >= 0])
        host_w = {int(e): (wlm.bf16_bits(d["W13"][e]), wlm.bf16_bits(d["W2"][e])) for e in touched}
        x_bits = wlm.bf16_bits(d["x"])
        samples.append(dict(wl=wl, tok=tok, ids=ids, w=d["w_np"], x=x_bits, host_w=host_w,
                            flops=6.0 * int(np.count_nonzero(ids[tok] >= 0)) * wl.H * wl.I))
        if host_cache is not None:
            host_cache[key] = dict(samples[-1])
    t0 = time.perf_counter()
    for s in samples:
        s["t"] = 0.0
    while True:
        for s in samples:
            ts = time.perf_counter()
            oracle.moe_forward_streamed(s["x"], s["ids"], s["w"], lambda e, hw=s["host_w"]: hw[e], s["wl"].E,
                                        s["tok"])
            dt = time.perf_counter() - ts
            s["t"] += dt
            t_total += dt
            flops_done += s["flops"]
        runs += 1
        if time.perf_counter() - t0 >= seconds:
            break
    sample_desc = "; ".join(f"{s['wl'].name}: {s['tok'].size}/{s['wl'].T} tokens" for s in samples)
    # per call at the full token count, scaled from the sample by tokens (the
    # oracle's work is per token): extrapolated, not measured at full size
    us_full = {s["wl"].name: s["t"] / runs * s["wl"].T / s["tok"].size * 1e6 for s in samples}
    return {"value": flops_done / t_total / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{sample_desc}; repeated {runs}x ({t_total:.1f} s of oracle time)",
            "seconds": t_total, "flops": flops_done,
            "us_per_call_extrapolated": us_full,
            "us_per_call_note": "extrapolated from the token sample to the full T"}


# ----------------------------------------------------------------------------- GPU arm

def make_inputs(names, device, experts=0, tokens=0):
    """Device inputs of the named workloads; experts/tokens > 0 shrink the
    workload (same per-expert shape) for small profiler captures."""
    import dataclasses
    out = []
    for n in names:
        wl = wlm.WORKLOADS[n]
        if experts > 0:
            wl = dataclasses.replace(wl, E=experts, name=f"{wl.name}_E{experts}")
        if tokens > 0:
            wl = dataclasses.replace(wl, T=tokens, name=f"{wl.name}_T{tokens}")
        ids_np, w_np = wlm.make_routing(wl)
        W13, W2 = wlm.make_weights(wl, device)
        d = dict(wl=wl, ids_np=ids_np, w_np=w_np, x=wlm.make_x(wl, device), W13=W13, W2=W2,
                 ids=torch.from_numpy(ids_np).to(device), w=torch.from_numpy(w_np).to(device))
        d["acct"] = call_accounting(wl, ids_np)
        out.append(d)
    return out


def prepare(B, names, device, args):
    """Device inputs, problems and caller buffers of the named batches."""
    inputs = make_inputs(names, device, args.experts, args.tokens)
    layout = (B.MOE_WEIGHTS_MXFP8 if args.weights == "mxfp8" else
              B.MOE_WEIGHTS_PACKED if args.packed else B.MOE_WEIGHTS_ROW_MAJOR)
    for d in inputs:
        wl = d["wl"]
        d["problem"] = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, path=args.path, weight_layout=layout,
                                      forward_form=args.form)
        if args.packed:   # model-load transform; the row-major copy is released
            d["W13"], d["W2"] = B.moe_pack_weights(d["problem"], d["W13"], d["W2"])
            torch.cuda.synchronize(device)
            torch.cuda.empty_cache()
        if args.weights == "mxfp8":   # quantized once at model load; the bf16 copy is released
            d["W13"], d["W2"] = B.moe_quantize_weights(d["problem"], d["W13"], d["W2"])
            torch.cuda.synchronize(device)
            torch.cuda.empty_cache()
            d["acct"] = call_accounting(wl, d["ids_np"], weight_bytes=33.0 / 32.0)
        d["bufs"] = B.Buffers(d["problem"], device)
        d["path"] = B.moe_resolve_path(d["problem"])
        d["profile"] = B.moe_resolve_profile(d["problem"])
    return inputs


def forward_step(B, inputs, stream, events=None):
    """One step: moe_forward over every batch of the workload (with stage events if given)."""
    for i, d in enumerate(inputs):
        b = d["bufs"]
        if events is None:
            B.moe_forward(d["problem"], d["x"], d["ids"], d["w"], d["W13"], d["W2"], b.expert_offsets, b.perm,
                          b.out, b.ws, stream=stream)
        else:
            B.moe_forward_profiled(d["problem"], d["x"], d["ids"], d["w"], d["W13"], d["W2"], b.expert_offsets,
                                   b.perm, b.out, b.ws, events[i], stream=stream)


def check_device_errors(B, inputs, stream):
    for d in inputs:
        err = B.moe_last_device_error(d["bufs"].ws, stream)
        if err:
            raise RuntimeError(f"device error word {err} on {d['wl'].name}")


def capture(stream, fn, steps: int):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for s in range(steps):
                fn(s)
    return g


def replay_timed(stream, graph, reps: int) -> float:
    """Milliseconds of `reps` back-to-back replays between two CUDA events on `stream`."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1)


def stage_profile(B, inputs, stream, steps: int = 4, reps: int = 2):
    """Stage times from a graph of `steps` steps of moe_forward_profiled (six
    events per forward, external event nodes between the kernels), replayed
    `reps` times; the stage times are those of the last replay. Returns
    (per-batch mean stage times in us, profiled step time in us)."""
    events = []
    for _ in range(steps):
        row = []
        for _ in inputs:
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
            for e in evs:
                e.record(stream)   # creates the underlying cudaEvent_t
            row.append(evs)
        events.append(row)
    stream.synchronize()
    g = capture(stream, lambda s: forward_step(B, inputs, stream, events[s]), steps)
    for _ in range(reps - 1):
        replay_timed(stream, g, 1)
    ms = replay_timed(stream, g, 1)
    stage_us = []
    for i in range(len(inputs)):
        per = np.array([[events[s][i][j].elapsed_time(events[s][i][j + 1]) * 1e3 for j in range(5)]
                        for s in range(steps)])
        stage_us.append(per.mean(axis=0))
    del g
    return stage_us, ms * 1e3 / steps


def tensor_peak(peaks: dict, region_s: float):
    """The measured bf16 peak that applies to a kernel timed over `region_s`
    seconds: the sustained figure (seconds-long loop under the power cap) for
    regions of a second or more, else the burst figure."""
    if region_s >= 1.0:
        return peaks["bf16_tflops_sustained"], f"bf16 dense, sustained ({peaks['source']}): timed region {region_s:.2f} s"
    return peaks["bf16_tflops"], f"bf16 dense, burst ({peaks['source']}): timed region {region_s * 1e3:.0f} ms < 1 s"


def dominant_kernel(inputs, stage_us, weights: str):
    """Which kernel dominates the step, its profiled time per step (us) and
    its algorithmic FLOPs and bytes per step. The gate-up GEMM holds 2/3 of
    the FLOPs and weight bytes; where both GEMMs run as one persistent kernel
    (M-small path) that kernel is timed as one, and where the whole forward is
    one kernel (decode-size batches) its stage marks all fall after it."""
    fused = all(d["profile"]["fused_mlp"] for d in inputs)
    mega = [d["profile"]["megakernel"] for d in inputs]

    def kernel_us(d, s):
        if d["profile"]["megakernel"]:
            return float(sum(s))
        return float(s[2]) + (float(s[3]) if fused else 0.0)

    us = sum(kernel_us(d, s) for d, s in zip(inputs, stage_us))
    flops = sum(d["acct"]["gemm1_flops"] * (1.5 if fused else 1.0) for d in inputs)
    nbytes = sum(d["acct"]["gemm1_bytes"] + (d["acct"]["gemm2_bytes"] if fused else 0.0) for d in inputs)
    if fused:
        name = ("fused_small_kernel (gate-up + down in one persistent launch"
                + ("; the whole forward for " + ", ".join(d["wl"].name for d, m in zip(inputs, mega) if m)
                   if any(mega) else "") + ")")
    else:
        paths = {d["path"][0] for d in inputs}
        name = ("grouped_gemm_pair_kernel (gate-up, CTA pairs, SiLU*up epilogue)" if paths == {1} else
                "grouped_gemm_kernel (gate-up, SiLU*up epilogue)")
    return {"name": name, "profiled_us": us, "flops": flops, "bytes": nbytes, "fused": fused,
            "key": traffic_key(inputs, weights, fused)}


def roofline_entry(kern: dict, kernel_us: float, peaks: dict, region_s: float, launches: int) -> dict:
    """roofline of the dominant kernel: algorithmic work per launch / its time per launch."""
    t_peak, t_kind = tensor_peak(peaks, region_s)
    t_tensor = kern["flops"] / (t_peak * 1e12)
    t_hbm = kern["bytes"] / (peaks["hbm_gbs"] * 1e9)
    per_launch_us = kernel_us / launches
    if t_tensor > t_hbm:
        alg = kern["flops"] / launches
        r = {"bound": "tensor", "achieved": alg / (per_launch_us * 1e-6) / 1e12, "peak": t_peak,
             "unit": "TFLOP/s", "peak_kind": t_kind}
        other = (peaks["bf16_tflops_sustained"] if t_peak == peaks["bf16_tflops"] else peaks["bf16_tflops"])
        r["frac_vs_other_bf16_peak"] = {"peak": other, "frac": r["achieved"] / other}
    else:
        alg = kern["bytes"] / launches
        r = {"bound": "hbm", "achieved": alg / (per_launch_us * 1e-6) / 1e9, "peak": peaks["hbm_gbs"],
             "unit": "GB/s", "peak_kind": f"HBM copy ({peaks['source']})"}
    r["frac"] = r["achieved"] / r["peak"]
    r["kernel"] = kern["name"]
    r["algorithmic_per_launch"] = alg
    r["algorithmic_bytes_per_launch"] = kern["bytes"] / launches
    r["kernel_us_per_launch"] = per_launch_us
    return r


def call_roofline(inputs, ms_per_step: float, peaks: dict, region_s: float) -> dict:
    """Whole-call roofline: per batch the slower of its FLOPs at the tensor
    peak and its touched bytes at the copy bandwidth, summed over the step."""
    t_peak, t_kind = tensor_peak(peaks, region_s)
    t_roof = 0.0
    bound = set()
    for d in inputs:
        tf = d["acct"]["flops"] / (t_peak * 1e12)
        tb = d["acct"]["bytes"] / (peaks["hbm_gbs"] * 1e9)
        t_roof += max(tf, tb)
        bound.add("tensor" if tf > tb else "hbm")
    return {"t_roof_us": t_roof * 1e6, "t_step_us": ms_per_step * 1e3, "frac": t_roof * 1e3 / ms_per_step,
            "bound": "+".join(sorted(bound)), "tensor_peak": t_peak, "tensor_peak_kind": t_kind,
            "hbm_peak_gbs": peaks["hbm_gbs"]}


def stage_dict(d, s):
    if d["profile"]["megakernel"]:
        return {"forward_one_kernel": float(sum(s))}
    return {k: float(v) for k, v in zip(STAGES, s)}


def run_ours(args, world, rank, local):
    from moe_routed_expert_routing_gb300.build import build
    build()
    from moe_routed_expert_routing_gb300 import binding as B

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    init_dist(world, local)
    inputs = prepare(B, WORKLOAD_SETS[args.workload], device, args)
    stream = torch.cuda.Stream(device)
    peaks = load_peaks()

    # warm-up: W steps in all. The first runs eagerly, outside capture (it sets
    # the kernels' function attributes); the rest replay the one-step graph
    # that the timed region replays, so its upload is warm too.
    with torch.cuda.stream(stream):
        forward_step(B, inputs, stream)
    stream.synchronize()
    check_device_errors(B, inputs, stream)
    graph = capture(stream, lambda s: forward_step(B, inputs, stream), 1)
    warmup = max(1, args.warmup)
    with torch.cuda.stream(stream):
        for _ in range(warmup - 1):
            graph.replay()
    stream.synchronize()

    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    barrier(world, device)
    torch.cuda.synchronize(device)
    clocks.start()
    time.sleep(0.25)
    clocks.mark_start()
    local_ms = replay_timed(stream, graph, args.steps)   # exactly K steps, one graph replay each
    torch.cuda.synchronize(device)
    clocks.mark_end()
    time.sleep(0.05)
    clk = clocks.stop()
    barrier(world, device)
    max_ms = max_over_ranks(local_ms, world, device)
    K = args.steps
    ms_per_step = max_ms / K
    check_device_errors(B, inputs, stream)

    # stage shares from the profiled graph (same steps, event nodes between
    # the kernels); the dominant kernel's time per step is its share of the
    # profiled step applied to the timed step, so it can never exceed it
    stage_us, prof_step_us = stage_profile(B, inputs, stream)
    kern = dominant_kernel(inputs, stage_us, args.weights)
    share = min(1.0, kern["profiled_us"] / prof_step_us)
    kernel_us = share * ms_per_step * 1e3
    region_s = max_ms * 1e-3
    roof = roofline_entry(kern, kernel_us, peaks, region_s, len(inputs))
    roof["kernel_time"] = (f"share {share:.4f} of the profiled step ({kern['profiled_us']:.1f} of "
                           f"{prof_step_us:.1f} us, CUDA events between the stages) times the timed step "
                           f"({ms_per_step * 1e3:.1f} us)")
    cap = NCU_TRAFFIC.get(kern["key"]) if kern["key"] else None
    traffic = None
    if cap and NCU_TRAFFIC["kernel_sha256"] == kernel_sha():
        traffic = cap["traffic"] / cap["algorithmic"] * roof["algorithmic_bytes_per_launch"]
    roof["traffic"] = traffic
    roof["traffic_note"] = (f"ncu dram read+write bytes per launch of {cap['case']}, scaled by algorithmic bytes"
                            if traffic is not None else "no capture for this kernel version/workload")

    flops_step = sum(d["acct"]["flops"] for d in inputs)
    bytes_step = sum(d["acct"]["bytes"] for d in inputs)
    value = world * flops_step * K / (max_ms * 1e-3) / 1e12
    e2e = run_e2e(B, inputs, stream, device, args, world)

    result = {
        "metric": "routed-MoE us/call & TFLOPS (dispatch+GEMMs+combine) vs roofline, 1 GB300",
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": " + ".join(d["wl"].describe() for d in inputs),
            "batches_per_step": [d["wl"].name for d in inputs],
            "paths": {d["wl"].name: {"path": {1: "tiled (CTA pairs)", 2: "small_m", 3: "tiled (1 CTA)"}[d["path"][0]],
                                     "tile_rows": d["path"][1]} for d in inputs},
            "l2": f"inputs larger than L2: {bytes_step / 1e9:.2f} GB of touched weights+activations per step",
            "timing": (f"one-step CUDA graph replayed {K}x between CUDA events (warm-up: 1 eager step + "
                       f"{warmup - 1} replays); stage times from a second graph of the same steps with stage "
                       f"events"),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "weights": ("MXFP8 (E4M3 codes + E8M0 scale per 32, expanded to bf16 on chip)"
                        if args.weights == "mxfp8" else "packed (access-ordered)" if args.packed else "row-major"),
        },
        "us_per_call": {d["wl"].name: float(sum(s)) * ms_per_step * 1e3 / prof_step_us
                        for d, s in zip(inputs, stage_us)},
        "us_per_call_note": ("each batch's share of the profiled step applied to the timed step; "
                             "us_per_call_alone: each batch timed in a graph of its own"),
        "us_per_call_alone": time_alone(B, inputs, stream),
        "profiled_ms_per_step": prof_step_us * 1e-3,
        "stages_us_profiled": {d["wl"].name: stage_dict(d, s) for d, s in zip(inputs, stage_us)},
        "tflops_per_step": flops_step / (ms_per_step * 1e-3) / 1e12,
        "call_roofline": call_roofline(inputs, ms_per_step, peaks, region_s),
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": sum(d["profile"]["kernel_launches"] for d in inputs) * K,
        "clocks": clk,
    }
    result["call_roofline"]["touched_expert_weights_gb"] = {
        d["wl"].name: d["acct"]["touched_experts"] * 3 * d["wl"].H * d["wl"].I
        * (33 / 32 if args.weights == "mxfp8" else 2) / 1e9 for d in inputs}
    if args.weights == "mxfp8":
        result["dtype"] = "bf16 (weights mxfp8)"
    cpu_inputs = inputs
    if rank == 0 and (args.packed or args.weights == "mxfp8"):
        result["cpu_baseline"] = None
        result["cpu_baseline_note"] = "not run with --packed / --weights mxfp8 (see the row-major bf16 line)"
    elif rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = time_oracle(cpu_inputs, args.cpu_seconds,
                                             tokens_cap=args.cpu_tokens if args.cpu_tokens > 0 else None)
        result["cpu_baseline"]["value_note"] = "oracle FLOP rate on the sample; a baseline, not the target"
    elif rank == 0:
        result["cpu_baseline"] = None
    # the other workloads of the same family, each timed on its own (one GPU only)
    if world == 1 and args.per_config and args.weights == "bf16":
        del inputs, cpu_inputs, graph
        torch.cuda.synchronize(device)
        torch.cuda.empty_cache()
        result["per_config"] = run_per_config(B, args, device, stream, peaks)
    return result


PER_CONFIG = ["prefill", "small", "decode"]


def time_alone(B, inputs, stream, target_ms: float = 60.0) -> dict:
    """µs per call of each batch of a multi-batch step, timed on its own: a
    graph of G calls of that batch alone (G * call >= ~5 ms), replayed so
    that ~target_ms of work sits between CUDA events, after two warm replays.
    (The stage shares of the profiled step overstate small batches: the event
    nodes between their kernels cut the launch overlap the timed graph has.)"""
    out = {}
    if len(inputs) < 2:
        return out
    for d in inputs:
        one = capture(stream, lambda s: forward_step(B, [d], stream), 1)
        replay_timed(stream, one, 2)
        est_ms = replay_timed(stream, one, 3) / 3
        G = max(1, min(50, int(math.ceil(5.0 / max(est_ms, 1e-3)))))
        g = capture(stream, lambda s: forward_step(B, [d], stream), G)
        reps = max(2, int(math.ceil(target_ms / (G * est_ms))))
        replay_timed(stream, g, 2)
        out[d["wl"].name] = replay_timed(stream, g, reps) * 1e3 / (reps * G)
        del one, g
    check_device_errors(B, inputs, stream)
    return out


def run_per_config(B, args, device, stream, peaks) -> dict:
    """us/call, TFLOP/s and the call-roofline fraction of each other workload:
    a graph of G steps (G * step >= ~10 ms) replayed so that ~args.config_ms of
    work is timed between CUDA events, after two warm replays."""
    out = {}
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[0]))
    clocks.start()
    for name in PER_CONFIG:
        if name == args.workload:
            continue
        inputs = prepare(B, WORKLOAD_SETS[name], device, args)
        with torch.cuda.stream(stream):
            forward_step(B, inputs, stream)
        stream.synchronize()
        check_device_errors(B, inputs, stream)
        one = capture(stream, lambda s: forward_step(B, inputs, stream), 1)
        replay_timed(stream, one, 2)
        est_ms = replay_timed(stream, one, 3) / 3
        G = max(1, min(20, int(math.ceil(10.0 / max(est_ms, 1e-3)))))
        g = capture(stream, lambda s: forward_step(B, inputs, stream), G)
        reps = max(2, int(math.ceil(args.config_ms / (G * est_ms))))
        replay_timed(stream, g, 2)
        ms = replay_timed(stream, g, reps)
        check_device_errors(B, inputs, stream)
        steps = reps * G
        ms_per_step = ms / steps
        stage_us, prof_step_us = stage_profile(B, inputs, stream)
        kern = dominant_kernel(inputs, stage_us, args.weights)
        share = min(1.0, kern["profiled_us"] / prof_step_us)
        region_s = ms * 1e-3
        roof = roofline_entry(kern, share * ms_per_step * 1e3, peaks, region_s, len(inputs))
        flops = sum(d["acct"]["flops"] for d in inputs)
        out[name] = {
            "workload": " + ".join(d["wl"].describe() for d in inputs),
            "steps": steps, "graph_steps": G,
            "ms_per_step": ms_per_step,
            "us_per_call": {d["wl"].name: float(sum(s)) * ms_per_step * 1e3 / prof_step_us
                            for d, s in zip(inputs, stage_us)},
            "us_per_call_alone": time_alone(B, inputs, stream),
            "tflops": flops / (ms_per_step * 1e-3) / 1e12,
            "call_roofline": call_roofline(inputs, ms_per_step, peaks, region_s),
            "dominant_kernel": {k: roof[k] for k in ("kernel", "bound", "achieved", "peak", "unit", "frac",
                                                       "kernel_us_per_launch")},
            "stages_us_profiled": {d["wl"].name: stage_dict(d, s) for d, s in zip(inputs, stage_us)},
            "paths": {d["wl"].name: d["profile"] for d in inputs},
        }
        del inputs, one, g
        torch.cuda.synchronize(device)
        torch.cuda.empty_cache()
    out["clocks"] = clocks.stop()
    return out


def run_e2e(B, inputs, stream, device, args, world):
    """Same metric through the public call, with every step's inputs copied
    from pinned host memory to the device and its outputs back, inside the
    timed region. A step's inputs of all batches (x, ids, weights) sit in one
    pinned staging buffer and go over in one copy; the outputs come back in
    one copy. The copies run on a stream of their own, double-buffered, as a
    serving loop overlaps them: step i+1's inputs go over while step i
    computes, and step i's outputs come back while step i+1 computes. The
    region ends when the last step's outputs are on the host."""
    def aligned(n):
        return (n + 255) // 256 * 256

    in_parts, out_parts = [], []
    o_in = o_out = 0
    for d in inputs:
        for name in ("x", "ids", "w"):
            t = d[name]
            in_parts.append((d, name, o_in, t))
            o_in += aligned(t.numel() * t.element_size())
        out_parts.append((d, o_out))
        o_out += aligned(d["bufs"].out.numel() * d["bufs"].out.element_size())
    host_in = torch.empty(o_in, dtype=torch.uint8).pin_memory()
    host_out = torch.empty(o_out, dtype=torch.uint8).pin_memory()
    dev_in = [torch.empty(o_in, dtype=torch.uint8, device=device) for _ in range(2)]
    dev_out = [torch.empty(o_out, dtype=torch.uint8, device=device) for _ in range(2)]
    views = [{}, {}]
    for d, name, off, t in in_parts:
        nbytes = t.numel() * t.element_size()
        host_in[off:off + nbytes].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
        for b in range(2):
            views[b][(id(d), name)] = dev_in[b][off:off + nbytes].view(t.dtype).view(t.shape)
    for d, off in out_parts:
        o = d["bufs"].out
        for b in range(2):
            views[b][(id(d), "out")] = dev_out[b][off:off + o.numel() * o.element_size()].view(o.dtype).view(o.shape)
    steps = max(1, min(args.steps, args.e2e_steps))
    h2d, d2h = o_in, o_out
    copy = torch.cuda.Stream(device)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]

    def h2d_copy(b):
        with torch.cuda.stream(copy):
            dev_in[b].copy_(host_in, non_blocking=True)
            ev_in[b].record(copy)

    def compute(b):
        stream.wait_event(ev_in[b])
        with torch.cuda.stream(stream):
            for d in inputs:
                v = views[b]
                B.moe_forward(d["problem"], v[(id(d), "x")], v[(id(d), "ids")], v[(id(d), "w")], d["W13"], d["W2"],
                              d["bufs"].expert_offsets, d["bufs"].perm, v[(id(d), "out")], d["bufs"].ws,
                              stream=stream)
            ev_done[b].record(stream)

    def d2h_copy(b):
        copy.wait_event(ev_done[b])
        with torch.cuda.stream(copy):
            host_out.copy_(dev_out[b], non_blocking=True)

    def run(n):
        # copy stream order: in(0); in(1), out(0); in(2), out(1); ... so that in(i+1)
        # follows out(i-1), which follows step i-1's compute: buffer i+1 % 2 is free
        h2d_copy(0)
        for i in range(n):
            compute(i % 2)
            if i + 1 < n:
                h2d_copy((i + 1) % 2)
            d2h_copy(i % 2)

    run(3)
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier(world, device)
    torch.cuda.synchronize(device)
    t0.record(copy)
    run(steps)
    t1.record(copy)
    torch.cuda.synchronize(device)
    ms = max_over_ranks(t0.elapsed_time(t1), world, device)
    # the last step's outputs, as the host received them, equal the timed graph's
    for d, off in out_parts:
        o = d["bufs"].out
        got = host_out[off:off + o.numel() * o.element_size()]
        if not torch.equal(got, o.contiguous().view(-1).view(torch.uint8).cpu()):
            raise RuntimeError(f"e2e output of {d['wl'].name} differs from the graph's")
    flops_step = sum(d["acct"]["flops"] for d in inputs)
    return {"value": world * flops_step * steps / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "ms_per_step": ms / steps,
            "api": "moe_forward (eager, C ABI); each step one pinned host->device copy of all its inputs and one "
                   "device->host copy of all its outputs, on a copy stream double-buffered against the compute "
                   "stream (step i+1's inputs and step i-1's outputs move while step i computes)"}


# ----------------------------------------------------------------------------- token sweep

SWEEP_TOKENS = [1, 8, 32, 128, 512, 2048, 8192]


def run_sweep(args, world, rank, local):
    """us/call vs roofline across token counts at one layer shape (E=384, k=6,
    H=7168, I=3072 by default): every batch shares the same weights, each gets
    its own routing; the launch profile follows from T alone."""
    from moe_routed_expert_routing_gb300.build import build
    build()
    from moe_routed_expert_routing_gb300 import binding as B
    import dataclasses

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    base = dataclasses.replace(wlm.WORKLOADS["prefill"], name="sweep")
    if args.experts > 0:
        base = dataclasses.replace(base, E=args.experts)
    W13, W2 = wlm.make_weights(base, device)
    peaks = load_peaks()
    stream = torch.cuda.Stream(device)
    rows = []
    for T in SWEEP_TOKENS:
        wl = dataclasses.replace(base, T=T, name=f"T{T}", seed=1000 + T)
        ids_np, w_np = wlm.make_routing(wl)
        x = wlm.make_x(wl, device)
        ids = torch.from_numpy(ids_np).to(device)
        w = torch.from_numpy(w_np).to(device)
        p = B.Problem.make(T, wl.E, wl.k, wl.H, wl.I, path=args.path, forward_form=args.form)
        bufs = B.Buffers(p, device)
        acct = call_accounting(wl, ids_np)

        def fwd():
            B.moe_forward(p, x, ids, w, W13, W2, bufs.expert_offsets, bufs.perm, bufs.out, bufs.ws, stream=stream)

        with torch.cuda.stream(stream):
            fwd()
        stream.synchronize()
        if B.moe_last_device_error(bufs.ws, stream):
            raise RuntimeError(f"device error at T={T}")
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for _ in range(GRAPH_STEPS):
                    fwd()
        reps = max(1, args.steps // GRAPH_STEPS)
        with torch.cuda.stream(stream):
            g.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize(device)
        us = e0.elapsed_time(e1) * 1e3 / (reps * GRAPH_STEPS)
        t_roof = max(acct["flops"] / (peaks["bf16_tflops_sustained"] * 1e12), acct["bytes"] / (peaks["hbm_gbs"] * 1e9))
        rows.append({"T": T, "us_per_call": us, "tflops": acct["flops"] / (us * 1e-6) / 1e12,
                     "touched_experts": acct["touched_experts"], "roof_us": t_roof * 1e6,
                     "roof_bound": "tensor" if acct["flops"] / (peaks["bf16_tflops_sustained"] * 1e12) >
                     acct["bytes"] / (peaks["hbm_gbs"] * 1e9) else "hbm",
                     "frac": t_roof * 1e6 / us, "profile": B.moe_resolve_profile(p)})
        del bufs, g
        torch.cuda.empty_cache()
    return {"sweep": "token count", "shape": f"E={base.E} k={base.k} H={base.H} I={base.I}, bf16, uniform routing",
            "steps_per_point": max(1, args.steps // GRAPH_STEPS) * GRAPH_STEPS, "rows": rows,
            "peaks": peaks}


def run_compare_forms(args, world, rank, local):
    """Decode-size forward as three kernels (MOE_FORWARD_SEPARATE) against one
    (MOE_FORWARD_ONE_KERNEL), per batch of the workload set: both captured as
    graphs of GRAPH_STEPS calls and replayed alternately in one process (an
    A/B in one process, as the DeepGEMM page measures its variants), median
    of 7 rounds of 20 replays. Not the bench line."""
    from moe_routed_expert_routing_gb300.build import build
    build()
    from moe_routed_expert_routing_gb300 import binding as B

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    forms = {"separate": B.MOE_FORWARD_SEPARATE, "one_kernel": B.MOE_FORWARD_ONE_KERNEL}
    layout = B.MOE_WEIGHTS_MXFP8 if args.weights == "mxfp8" else B.MOE_WEIGHTS_ROW_MAJOR
    rows = []
    for name in WORKLOAD_SETS[args.workload]:
        d = make_inputs([name], device, args.experts, args.tokens)[0]
        wl = d["wl"]
        if layout == B.MOE_WEIGHTS_MXFP8:
            q = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, path=args.path, weight_layout=layout)
            d["W13"], d["W2"] = B.moe_quantize_weights(q, d["W13"], d["W2"])
            torch.cuda.synchronize(device)
            torch.cuda.empty_cache()
        graphs, bufs = {}, {}
        for f, code in forms.items():
            p = B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, path=args.path, forward_form=code, weight_layout=layout)
            bufs[f] = B.Buffers(p, device)

            def fwd(p=p, b=bufs[f]):
                B.moe_forward(p, d["x"], d["ids"], d["w"], d["W13"], d["W2"], b.expert_offsets, b.perm, b.out,
                              b.ws, stream=stream)

            with torch.cuda.stream(stream):
                fwd()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                with torch.cuda.graph(g, stream=stream):
                    for _ in range(GRAPH_STEPS):
                        fwd()
            graphs[f] = g
        us = {f: [] for f in forms}
        for _ in range(7):
            for f, g in graphs.items():
                with torch.cuda.stream(stream):
                    for _ in range(2):
                        g.replay()
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    for _ in range(20):
                        g.replay()
                    e1.record(stream)
                torch.cuda.synchronize(device)
                us[f].append(e0.elapsed_time(e1) * 1e3 / (20 * GRAPH_STEPS))
        for f in forms:
            if B.moe_last_device_error(bufs[f].ws, stream):
                raise RuntimeError(f"device error ({f}) on {name}")
        same = torch.equal(bufs["separate"].out.view(torch.int16), bufs["one_kernel"].out.view(torch.int16))
        rows.append({"workload": wl.describe(), "us_per_call": {f: float(np.median(v)) for f, v in us.items()},
                     "rounds_us": {f: [round(x, 2) for x in v] for f, v in us.items()},
                     "bit_identical": bool(same), "weights": args.weights,
                     "auto_picks": "one_kernel" if B.moe_resolve_profile(
                         B.Problem.make(wl.T, wl.E, wl.k, wl.H, wl.I, path=args.path, weight_layout=layout))[
                             "megakernel"] else "separate"})
        del graphs, bufs, d
        torch.cuda.empty_cache()
    return {"compare": "moe_forward forms (separate kernels vs one kernel)", "rows": rows}


# ----------------------------------------------------------------------------- reference arm

def run_reference(args, world, rank, local):
    """The CPU oracle as the reference arm: same workload, metric and unit."""
    names = WORKLOAD_SETS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    if dev == "cuda":
        torch.cuda.set_device(local)
    inputs = make_inputs(names, dev, args.experts, args.tokens)
    # size each step so that warmup + steps finish within ~2 minutes
    budget = max(0.02, 120.0 / (args.steps + args.warmup))
    calib = time_oracle(inputs, 0.0, tokens_cap=1)
    per_token = calib["seconds"] / max(1, len(inputs))
    tokens = max(1, int(budget / max(per_token * len(inputs), 1e-9)))
    cache = {}
    for _ in range(args.warmup):
        time_oracle(inputs, 0.0, tokens_cap=tokens, host_cache=cache)
    flops, secs = 0.0, 0.0
    us_full = {}
    for _ in range(args.steps):
        r = time_oracle(inputs, 0.0, tokens_cap=tokens, host_cache=cache)
        flops += r["flops"]
        secs += r["seconds"]
        for name, us in r["us_per_call_extrapolated"].items():
            us_full[name] = us_full.get(name, 0.0) + us / args.steps
    value = flops / secs / 1e12
    full_flops = sum(d["acct"]["flops"] for d in inputs)
    ms_per_step = full_flops / (value * 1e12) * 1e3
    return {
        "impl": "reference",
        "metric": "routed-MoE us/call & TFLOPS (dispatch+GEMMs+combine) vs roofline, 1 GB300",
        "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": " + ".join(d["wl"].describe() for d in inputs),
                   "note": "ms_per_step extrapolated to the full step from the oracle's FLOP rate"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": r["cores"], "kind": "oracle",
                         "sample": f"each step, at most {tokens} token(s) of each batch ({r['sample']})",
                         "us_per_call_extrapolated": us_full, "us_per_call_note": r["us_per_call_note"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- main

def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_SETS), default="large")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="skip the per-config block (prefill, small, decode timed on their own)")
    ap.add_argument("--config-ms", type=float, default=150.0,
                    help="milliseconds of work timed per entry of the per-config block")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-tokens", type=int, default=0, help="tokens per batch in the CPU sample (0 = auto)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--experts", type=int, default=0, help="override E (small profiler cases)")
    ap.add_argument("--tokens", type=int, default=0, help="override T (small profiler cases)")
    ap.add_argument("--packed", action="store_true", help="weights in the access-ordered PACKED layout")
    ap.add_argument("--sweep", action="store_true", help="token-count sweep at the 384-expert shape (not the bench line)")
    ap.add_argument("--path", type=int, default=0, choices=[0, 1, 2, 3],
                    help="expert-GEMM path: 0 auto, 1 tiled CTA pairs, 2 M-small, 3 tiled single CTA")
    ap.add_argument("--weights", choices=["bf16", "mxfp8"], default="bf16",
                    help="expert weights: bf16, or MXFP8 quantized at load (M-small path only)")
    ap.add_argument("--form", type=int, default=0, choices=[0, 1, 2],
                    help="decode-size forward: 0 auto, 1 separate kernels, 2 one kernel")
    ap.add_argument("--compare-forms", action="store_true",
                    help="decode-size forward: separate kernels vs one kernel, alternating (not the bench line)")
    return ap.parse_args(argv)


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_env()
    if args.steps < 1 or args.warmup < 0:
        raise SystemExit("--steps must be >= 1 and --warmup >= 0")
    if args.impl == "reference":
        if rank != 0:
            return 0
        if args.cpu_tokens == 0:
            args.cpu_tokens = 1
        line = run_reference(args, world, rank, local)
        print(json.dumps(line), flush=True)
        return 0
    if args.sweep:
        if rank == 0:
            print(json.dumps(run_sweep(args, world, rank, local)), flush=True)
        return 0
    if args.compare_forms:
        if rank == 0:
            print(json.dumps(run_compare_forms(args, world, rank, local)), flush=True)
        return 0
    if args.cpu_tokens == 0:
        wl_T = max(wlm.WORKLOADS[n].T for n in WORKLOAD_SETS[args.workload])
        args.cpu_tokens = wl_T if wl_T <= 8 else 16
    line = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
