"""The oracle and the CUDA path share no code (host only).

* the package (binding, build, CUDA sources) never imports or includes the
  oracle;
* the oracle never imports the package and includes only system headers;
* the seeded input generators (``workloads.py``) import neither;
* ``bench.py`` reaches the oracle only from ``time_oracle``, its CPU-baseline
  and reference legs, never at module level or on the GPU legs.
"""
from __future__ import annotations

import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = "moe_routed_expert_routing_gb300"


def _imported_roots(tree: ast.AST) -> set:
    roots = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            roots.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            roots.add(node.module.split(".")[0])
    return roots


def _parse(path: str) -> ast.AST:
    with open(path) as f:
        return ast.parse(f.read(), filename=path)


def _local_includes(path: str) -> list:
    with open(path) as f:
        return re.findall(r'^\s*#\s*include\s+"([^"]+)"', f.read(), flags=re.M)


def test_package_never_reaches_the_oracle():
    for dirpath, _, files in os.walk(os.path.join(ROOT, PKG)):
        for name in files:
            path = os.path.join(dirpath, name)
            if name.endswith(".py"):
                assert "oracle" not in _imported_roots(_parse(path)), path
            elif name.endswith((".cu", ".cuh", ".h")):
                for inc in _local_includes(path):
                    assert "oracle" not in inc, (path, inc)


def test_oracle_never_reaches_the_package():
    odir = os.path.join(ROOT, "oracle")
    for name in os.listdir(odir):
        path = os.path.join(odir, name)
        if name.endswith(".py"):
            roots = _imported_roots(_parse(path))
            assert PKG not in roots and "bench" not in roots and "workloads" not in roots, path
        elif name.endswith((".c", ".h")):
            assert _local_includes(path) == [], path     # system headers only


def test_input_generators_import_neither_side():
    roots = _imported_roots(_parse(os.path.join(ROOT, "workloads.py")))
    assert "oracle" not in roots and PKG not in roots


class _ImportSites(ast.NodeVisitor):
    """Every import of ``root``, with the innermost function around it
    (None at module level)."""

    def __init__(self, root: str):
        self.root, self.stack, self.sites = root, [], []

    def _fn(self, node):
        self.stack.append(node.name)
        self.generic_visit(node)
        self.stack.pop()

    visit_FunctionDef = visit_AsyncFunctionDef = _fn

    def visit_Import(self, node):
        if any(a.name.split(".")[0] == self.root for a in node.names):
            self.sites.append(self.stack[-1] if self.stack else None)

    def visit_ImportFrom(self, node):
        if node.module and node.level == 0 and node.module.split(".")[0] == self.root:
            self.sites.append(self.stack[-1] if self.stack else None)


def _oracle_import_sites(source: str) -> set:
    v = _ImportSites("oracle")
    v.visit(ast.parse(source))
    return set(v.sites)


def test_bench_reaches_the_oracle_only_from_its_cpu_leg():
    with open(os.path.join(ROOT, "bench.py")) as f:
        assert _oracle_import_sites(f.read()) == {"time_oracle"}
    # the check itself bites: a nested import elsewhere, or one at module level
    assert _oracle_import_sites("def main():\n    if True:\n        import oracle\n") == {"main"}
    assert _oracle_import_sites("from oracle import load\n") == {None}
