"""Structural rules between the CUDA path, the CPU oracle and the shared
input generators, checked on the source files: the product never reaches the
oracle, the oracle shares no code with the CUDA path, the generators hold no
arithmetic of either, and a missing library is an error, not a fallback."""
import ast
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "lazy_sparse_attention_token_b300")


def _read(path):
    with open(path) as f:
        return f.read()


def _py_files(d):
    for dirpath, _, files in os.walk(d):
        if "__pycache__" in dirpath or "_build" in dirpath:
            continue
        for f in files:
            if f.endswith(".py"):
                yield os.path.join(dirpath, f)


def _imports(path):
    tree = ast.parse(_read(path), path)
    out = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            out.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            out.add(node.module.split(".")[0])
    return out


def test_package_never_imports_the_oracle():
    files = list(_py_files(PKG))
    assert files
    for f in files:
        assert "oracle" not in _imports(f), f
    for f in os.listdir(os.path.join(PKG, "csrc")):
        text = _read(os.path.join(PKG, "csrc", f))
        assert "oracle" not in text.lower(), f


def test_oracle_shares_no_code_with_the_cuda_path():
    odir = os.path.join(ROOT, "oracle")
    for f in _py_files(odir):
        imps = _imports(f)
        assert "lazy_sparse_attention_token_b300" not in imps and "synth" not in imps, f
    for f in os.listdir(odir):
        if f.endswith((".c", ".h")):
            for inc in re.findall(r'#include\s*[<"]([^>"]+)[>"]', _read(os.path.join(odir, f))):
                assert "/" not in inc and not inc.endswith((".cuh", ".cu")) and inc != "flashloop.h", (f, inc)


def test_input_generators_import_neither_side():
    for f in _py_files(os.path.join(ROOT, "synth")):
        imps = _imports(f)
        assert "oracle" not in imps and "lazy_sparse_attention_token_b300" not in imps, f


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    import lazy_sparse_attention_token_b300.flashloop as F
    monkeypatch.setattr(F, "_lib", None)
    monkeypatch.setattr(F, "LIB_PATH", str(tmp_path / "libflashloop.so"))
    with pytest.raises(FileNotFoundError):
        F.lib()


def test_bench_reaches_the_oracle_only_through_its_cpu_legs():
    """In bench.py only the cpu_baseline leg and the reference arm may run the
    oracle: every function that uses it (directly, or through a helper that
    does) is called only from those two or from another such helper."""
    tree = ast.parse(_read(os.path.join(ROOT, "bench.py")))
    funcs = {n.name: n for n in tree.body if isinstance(n, ast.FunctionDef)}

    def names(fn):
        return {n.id for n in ast.walk(fn) if isinstance(n, ast.Name)} | \
               {a.name.split(".")[0] for n in ast.walk(fn) if isinstance(n, ast.Import) for a in n.names} | \
               {n.module.split(".")[0] for n in ast.walk(fn) if isinstance(n, ast.ImportFrom) and n.module}

    top = {a.name.split(".")[0] for n in tree.body if isinstance(n, ast.Import) for a in n.names} | \
          {n.module.split(".")[0] for n in tree.body if isinstance(n, ast.ImportFrom) and n.module}
    assert "oracle" not in top
    legs = {"cpu_baseline", "reference"}
    # helpers: functions other than the legs that use the oracle, directly or by
    # calling another helper
    helpers = {f for f, n in funcs.items() if f not in legs and "oracle" in names(n)}
    changed = True
    while changed:
        changed = False
        for f, n in funcs.items():
            if f not in legs and f not in helpers and names(n) & helpers:
                helpers.add(f)
                changed = True
    for leg in legs:   # both legs do run the oracle
        assert "oracle" in names(funcs[leg]) or names(funcs[leg]) & helpers, leg
    # the timed paths and the entry point reach the oracle only by calling a leg
    for f in ("native", "native_decode", "e2e_leg", "main"):
        assert f not in helpers, f
