"""Build libmoe.so in-tree for sm_103a (GB300) with nvcc.

The translation units compile in parallel (one ``-gencode``, no cmake), then
link into ``moe_routed_expert_routing_gb300/_build/libmoe.so`` against the
shared CUDA runtime (the same libcudart.so.13 PyTorch loads).

``python -m moe_routed_expert_routing_gb300.build [--force]``
"""
from __future__ import annotations

import concurrent.futures as cf
import fcntl
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
INCLUDE = os.path.join(ROOT, "include")
SOURCES = ["moe_api.cu", "dispatch.cu", "dispatch_noalloc.cu", "combine.cu", "grouped_gemm.cu", "weights_pack.cu",
           "weights_mx.cu"]
HEADERS = ["ptx.cuh", "moe_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def lib_path() -> str:
    return os.path.join(BUILD, "libmoe.so")


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: libmoe.so cannot be built")
    return cand


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile what is stale and link. Several processes (one per rank) may call
    this at once: a file lock lets the first build and the others find it done."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    with open(os.path.join(BUILD, ".build.lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        return _build_locked(nvcc, force, verbose, extra_flags)


def _build_locked(nvcc: str, force: bool, verbose: bool, extra_flags) -> str:
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "moe.h")]
    common = ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
              "--expt-relaxed-constexpr", *extra_flags]
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s, *hdrs]):
            jobs.append([nvcc, *common, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        list(ex.map(run, jobs))
    out = lib_path()
    if force or jobs or _stale(out, objs):
        tmp = out + f".tmp{os.getpid()}"
        run([nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs])
        os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
