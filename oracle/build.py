"""Build step for the C oracle (test infrastructure; see oracle/__init__.py).

``python -m oracle.build`` compiles ``moe_oracle.c`` into
``oracle/_build/liboracle.so`` with gcc. Plain portable C: it builds the same
on x86_64 and aarch64 and ``-ffp-contract=off`` keeps results bit-identical
across the two.
"""
from __future__ import annotations

import os
import subprocess
import sys

_HERE = os.path.dirname(os.path.abspath(__file__))


def oracle_lib_path() -> str:
    return os.path.join(_HERE, "_build", "liboracle.so")


def build_oracle(force: bool = False) -> str:
    src = os.path.join(_HERE, "moe_oracle.c")
    out = oracle_lib_path()
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build_oracle(force="--force" in sys.argv))
