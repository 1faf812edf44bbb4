"""The oracle and the CUDA path share no code, and the product path never reaches the oracle (CPU).

The product package (the binding, its build, the CUDA sources) must not import, include or link anything
under ``oracle/``; the oracle must not import the package or include its headers. Only the seeded input
generator (``synth``) serves both, from the tests.
"""
import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "speculative_decoding_verification_35_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _files(top, exts):
    for d, _, names in os.walk(top):
        if "__pycache__" in d:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def _imported_modules(path):
    tree = ast.parse(open(path, encoding="utf-8").read())
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            yield from (a.name for a in node.names)
        elif isinstance(node, ast.ImportFrom):
            yield ("." * node.level) + (node.module or "")


def test_product_package_never_imports_the_oracle():
    for f in _files(PKG, (".py",)):
        for m in _imported_modules(f):
            assert m.split(".")[0] != "oracle", (f, m)


def test_cuda_sources_never_include_oracle_code():
    for f in _files(os.path.join(PKG, "csrc"), (".cu", ".cuh", ".h")):
        for inc in re.findall(r'#include\s+["<]([^">]+)[">]', open(f, encoding="utf-8").read()):
            assert "oracle" not in inc and "verify_ref" not in inc, (f, inc)


def test_oracle_never_imports_the_package_or_its_headers():
    for f in _files(ORACLE, (".py",)):
        for m in _imported_modules(f):
            assert "speculative_decoding" not in m and "specverify" not in m, (f, m)
    for f in _files(ORACLE, (".c", ".h")):
        for inc in re.findall(r'#include\s+["<]([^">]+)[">]', open(f, encoding="utf-8").read()):
            assert not inc.startswith("sv_") and "specverify" not in inc, (f, inc)
