"""The product path and the oracle stay apart (CPU, static): nothing in the package or
its CUDA sources imports, includes or loads the oracle; the oracle imports nothing
from the package; the shared input generators hold no attention arithmetic that the
oracle could borrow; and the product fails loudly when its library is missing."""
import ast
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "paged_kv_cache_90_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _files(top, exts):
    for d, dirs, names in os.walk(top):
        dirs[:] = [x for x in dirs if not x.startswith(("_build", "__pycache__"))]
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def _imported_modules(path):
    with open(path) as f:
        tree = ast.parse(f.read(), path)
    mods = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            mods.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom):
            if node.level == 0 and node.module:
                mods.add(node.module.split(".")[0])
    return mods


def test_package_never_imports_the_oracle():
    for path in _files(PKG, (".py",)):
        assert "oracle" not in _imported_modules(path), path
        with open(path) as f:
            text = f.read()
        assert "liboracle" not in text and "paged_ref" not in text, path


def test_cuda_sources_include_nothing_of_the_oracle():
    for path in _files(os.path.join(PKG, "csrc"), (".cu", ".cuh", ".h")):
        with open(path) as f:
            includes = re.findall(r'#include\s+[<"]([^>"]+)[>"]', f.read())
        assert not any("oracle" in i or "paged_ref" in i for i in includes), path


def test_oracle_imports_nothing_of_the_package():
    for path in _files(ORACLE, (".py",)):
        assert "paged_kv_cache_90_gb300" not in _imported_modules(path), path
    with open(os.path.join(ORACLE, "paged_ref.c")) as f:
        includes = re.findall(r'#include\s+[<"]([^>"]+)[>"]', f.read())
    assert all(i in {"math.h", "stdint.h", "stdlib.h", "string.h", "omp.h"} for i in includes), includes


def test_input_generators_hold_no_attention_arithmetic():
    """The one module both sides use draws inputs; softmax, log-sum-exp and products of
    queries with keys belong to the two implementations only.  (Its one exponential
    draws lognormal context lengths.)"""
    with open(os.path.join(PKG, "workloads.py")) as f:
        tree = ast.parse(f.read())
    banned = {"softmax", "log_softmax", "logsumexp", "exp2", "einsum", "matmul", "bmm", "mm", "dot",
              "scaled_dot_product_attention"}
    exps = 0
    for node in ast.walk(tree):
        assert not (isinstance(node, ast.BinOp) and isinstance(node.op, ast.MatMult)), "matrix product"
        if isinstance(node, ast.Call):
            f = node.func
            name = f.attr if isinstance(f, ast.Attribute) else f.id if isinstance(f, ast.Name) else ""
            assert name not in banned, name
            exps += name == "exp"
    assert exps == 1


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    from paged_kv_cache_90_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        binding.load_library(str(tmp_path / "libpkv.so"))
