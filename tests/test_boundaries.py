"""The product never routes through the oracle and has no CPU fallback (no GPU):
the package does not import `oracle`, bench.py imports it only inside its CPU
baseline / reference legs, and the binding raises when libbsa.so is missing."""
import ast
import os

import pytest

from dynamic_block_sparse_mean_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "dynamic_block_sparse_mean_gb300")


def _imports(tree):
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield node, a.name
        elif isinstance(node, ast.ImportFrom):
            yield node, node.module or ""


def test_package_never_imports_the_oracle():
    for name in sorted(os.listdir(PKG)):
        if name.endswith(".py"):
            tree = ast.parse(open(os.path.join(PKG, name)).read())
            for _, mod in _imports(tree):
                assert not mod.split(".")[0] == "oracle", (name, mod)
    for name in sorted(os.listdir(os.path.join(PKG, "csrc"))):
        for line in open(os.path.join(PKG, "csrc", name)):
            if line.lstrip().startswith("#include"):
                assert "oracle" not in line, (name, line)


def test_bench_imports_the_oracle_only_in_its_cpu_legs():
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    allowed = {"oracle_rows", "cpu_oracle_throughput", "run_reference"}
    for fn in ast.walk(tree):
        if isinstance(fn, (ast.FunctionDef, ast.AsyncFunctionDef)):
            for node, mod in _imports(fn):
                if mod.split(".")[0] == "oracle":
                    assert fn.name in allowed, fn.name
    for node in tree.body:                         # nothing at module level
        if isinstance(node, (ast.Import, ast.ImportFrom)):
            names = [a.name for a in node.names] if isinstance(node, ast.Import) else [node.module]
            assert all((n or "").split(".")[0] != "oracle" for n in names)


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(_lib, "LIB_PATH", os.path.join(PKG, "no_such_libbsa.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _lib.lib()
