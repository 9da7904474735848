"""The oracle and the CUDA path share no code.  The product package (its
Python modules and CUDA sources) never imports or includes anything from
oracle/, and the oracle imports nothing from the product package.  Only the
tests, the smoke check and the benchmark's CPU legs use the oracle."""
import ast
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = "routing_dispatch_expert_05_b300"


def _imports(path):
    """Every module name imported anywhere in a file (top level or inside
    functions)."""
    tree = ast.parse(open(path).read())
    names = []
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names += [a.name for a in node.names]
        elif isinstance(node, ast.ImportFrom):
            names.append(("." * node.level) + (node.module or ""))
    return names


def test_product_never_imports_the_oracle():
    files = glob.glob(os.path.join(ROOT, PKG, "**", "*.py"), recursive=True)
    assert files
    for f in files:
        for name in _imports(f):
            assert not name.split(".")[0].lstrip(".") == "oracle", (f, name)
            assert "oracle" not in name, (f, name)


def test_cuda_sources_include_nothing_from_the_oracle():
    files = glob.glob(os.path.join(ROOT, PKG, "csrc", "*"))
    assert files
    for f in files:
        for line in open(f):
            if re.match(r"\s*#\s*include", line):
                assert "oracle" not in line, (f, line)


def test_oracle_imports_nothing_from_the_product():
    files = glob.glob(os.path.join(ROOT, "oracle", "*.py"))
    assert files
    for f in files:
        for name in _imports(f):
            assert not name.startswith(PKG), (f, name)
            assert name.split(".")[0] in ("numpy", "oracle", "__future__", "math",
                                          "dataclasses", "typing", ""), (f, name)
