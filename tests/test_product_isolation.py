"""The product path stands alone: the package and the C sources neither
import nor include the oracle (test infrastructure) or anything outside the
tree, and the binding fails loudly, with no fallback, when the library it
wraps is missing."""

import ast
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "sparse_attention_indexer_pmqa_gb300")


def _py_imports(path):
    tree = ast.parse(open(path).read(), filename=path)
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            names.add(node.module.split(".")[0])
    return names


def test_package_python_does_not_import_the_oracle_or_the_generators():
    for name in os.listdir(PKG):
        if name.endswith(".py"):
            imports = _py_imports(os.path.join(PKG, name))
            assert not imports & {"oracle", "synth", "tests", "bench"}, (name, imports)


def test_cuda_sources_include_only_their_own_headers_and_the_toolkit():
    csrc = os.path.join(PKG, "csrc")
    for name in os.listdir(csrc):
        if name.endswith((".cu", ".cuh")):
            for inc in re.findall(r'#include\s+"([^"]+)"', open(os.path.join(csrc, name)).read()):
                target = os.path.normpath(os.path.join(csrc, inc))
                assert target.startswith(csrc) or target == os.path.join(ROOT, "include", "pmqa.h"), \
                    (name, inc)


def test_binding_raises_when_the_library_is_missing(tmp_path):
    from sparse_attention_indexer_pmqa_gb300 import pmqa

    saved = pmqa._lib
    pmqa._lib = None
    try:
        with pytest.raises(FileNotFoundError):
            pmqa.load(str(tmp_path / "libpmqa.so"))
    finally:
        pmqa._lib = saved
