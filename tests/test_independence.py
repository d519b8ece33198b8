"""The oracle and the CUDA path stay apart: the library package and the C
header never name the oracle, the oracle never imports the library or its
build, the library's link line names no oracle object, and the benchmark
imports the oracle only inside its CPU-baseline leg and its reference arm.
The seeded generators (`synth/`) are the one module both sides use."""
import ast
import glob
import os

import pytest


def _read(path):
    with open(path) as f:
        return f.read()


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _files(sub, exts):
    out = []
    for ext in exts:
        out += glob.glob(os.path.join(ROOT, sub, "**", "*" + ext), recursive=True)
    return [f for f in out if "_build" not in f and "__pycache__" not in f]


def test_product_sources_never_name_the_oracle():
    srcs = _files("quantized_expert_cache_gb300", (".py", ".cu", ".cuh", ".h", ".cpp")) + _files("include", (".h",))
    assert srcs
    for f in srcs:
        text = _read(f).lower()
        assert "oracle" not in text, f


def test_oracle_does_not_import_the_library():
    for f in _files("oracle", (".py", ".c", ".h")):
        text = _read(f)
        assert "quantized_expert_cache_gb300" not in text, f
        assert "libmoecache" not in text, f
        assert "csrc" not in text, f


def test_generators_hold_no_library_or_oracle_code():
    for f in _files("synth", (".py", ".c", ".h")):
        text = _read(f)
        assert "quantized_expert_cache_gb300" not in text and "libmoecache" not in text, f
        for line in text.splitlines():
            s = line.strip()
            if s.startswith(("import ", "from ", "#include")):
                assert "oracle" not in s, (f, s)


@pytest.mark.parametrize("script", ["bench.py", "__graft_entry__.py"])
def test_oracle_imported_only_by_the_allowed_functions(script):
    allowed = {"bench.py": {"cpu_baseline", "run_reference"}, "__graft_entry__.py": {"build", "smoke"}}[script]
    tree = ast.parse(_read(os.path.join(ROOT, script)))
    found = []

    def visit(node, fn):
        for child in ast.iter_child_nodes(node):
            name = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else fn
            if isinstance(child, ast.Import):
                if any(a.name.split(".")[0] == "oracle" for a in child.names):
                    found.append(name)
            elif isinstance(child, ast.ImportFrom):
                if (child.module or "").split(".")[0] == "oracle":
                    found.append(name)
            visit(child, name)

    visit(tree, None)
    assert found, script
    assert set(found) <= allowed, (script, found)


def test_library_link_line_names_no_oracle_object():
    from quantized_expert_cache_gb300 import build as b

    src = _read(b.__file__)
    assert "oracle" not in src.lower()
    # every translation unit and header the library compiles is in its csrc/
    for s in b.SOURCES + b.HEADERS:
        assert os.path.basename(s) == s and os.path.exists(os.path.join(b.CSRC, s)), s
    assert os.path.dirname(b.CSRC) == os.path.join(ROOT, "quantized_expert_cache_gb300")
