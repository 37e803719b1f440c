"""The oracle and the CUDA path stay apart, and the product has no fallback (CPU, static).

- No file of the library (the package's Python and its CUDA/C++ sources, the public header)
  names the oracle, and no file of the oracle names the library or its sources.
- bench.py and __graft_entry__.py import the oracle only inside the functions that may use it:
  the bench's CPU-baseline and reference legs (through `_oracle_sample` / `_oracle_workloads`,
  called from the rank-0 CPU baseline and from `run_reference` alone), and the entry point's
  `build()` (which compiles it) and `smoke()` (which checks against it).
- With libkda.so absent, the binding raises on its first call instead of computing anything.
"""
import ast
import os
import re

import pytest

import kda_state_chunked_gb300 as kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "kda_state_chunked_gb300")
ORACLE = os.path.join(ROOT, "oracle")
SRC_EXT = (".py", ".cu", ".cuh", ".cpp", ".h", ".c")


def _files(top):
    for dirpath, dirnames, filenames in os.walk(top):
        dirnames[:] = [d for d in dirnames if not d.startswith(("_build", "__pycache__"))]
        for f in filenames:
            if f.endswith(SRC_EXT):
                yield os.path.join(dirpath, f)


def test_library_sources_never_name_the_oracle():
    """C/CUDA sources and the header never mention it; the package's Python never imports or
    references it (the seeded input module may say in its docstring that both sides use it)."""
    files = list(_files(PKG)) + [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))]
    native = [f for f in files if not f.endswith(".py")]
    python = [f for f in files if f.endswith(".py")]
    assert len(native) > 10 and len(python) >= 4
    pat = re.compile(r"\boracle\b")
    assert [f for f in native if pat.search(open(f, encoding="utf-8").read())] == []
    bad = []
    for f in python:
        tree = ast.parse(open(f, encoding="utf-8").read())
        for node in ast.walk(tree):
            if isinstance(node, ast.Import) and any("oracle" in a.name for a in node.names):
                bad.append((f, node.lineno))
            if isinstance(node, ast.ImportFrom) and "oracle" in (node.module or ""):
                bad.append((f, node.lineno))
            if isinstance(node, ast.Name) and node.id == "oracle":
                bad.append((f, node.lineno))
            if isinstance(node, ast.Constant) and isinstance(node.value, str) and "oracle/" in node.value:
                bad.append((f, node.lineno))
    assert bad == []


def _without_module_docstring(text):
    """Python source minus its module docstring (which may say, in prose, that the library is
    a separate thing)."""
    tree = ast.parse(text)
    if tree.body and isinstance(tree.body[0], ast.Expr) and isinstance(getattr(tree.body[0], "value", None), ast.Constant):
        lines = text.splitlines(keepends=True)
        return "".join(lines[tree.body[0].end_lineno:])
    return text


def test_oracle_sources_never_name_the_library():
    files = list(_files(ORACLE))
    assert any(f.endswith(".c") for f in files) and any(f.endswith(".py") for f in files)
    pat = re.compile(r"kda_state_chunked_gb300|csrc|libkda|kda\.h|sm100_ptx|tc_common")
    bad = []
    for f in files:
        text = open(f, encoding="utf-8").read()
        if f.endswith(".py"):
            text = _without_module_docstring(text)
        if pat.search(text):
            bad.append(f)
    assert bad == []


def _oracle_imports(path):
    """[(top-level function enclosing the import or None, line)] of every oracle import."""
    tree = ast.parse(open(path, encoding="utf-8").read())
    out = []
    for top in tree.body:
        owner = top.name if isinstance(top, (ast.FunctionDef, ast.AsyncFunctionDef)) else None
        for node in ast.walk(top):
            if isinstance(node, ast.Import) and any(a.name.split(".")[0] == "oracle" for a in node.names):
                out.append((owner, node.lineno))
            if isinstance(node, ast.ImportFrom) and (node.module or "").split(".")[0] == "oracle":
                out.append((owner, node.lineno))
    return out


def _callers(path, names):
    """Top-level functions of a file that call any of `names`."""
    tree = ast.parse(open(path, encoding="utf-8").read())
    out = set()
    for top in tree.body:
        for node in ast.walk(top):
            if isinstance(node, ast.Call) and isinstance(node.func, ast.Name) and node.func.id in names:
                out.add(top.name if isinstance(top, ast.FunctionDef) else None)
    return out


def test_bench_uses_the_oracle_only_in_its_cpu_legs():
    path = os.path.join(ROOT, "bench.py")
    owners = {o for o, _ in _oracle_imports(path)}
    assert owners == {"_oracle_sample", "_oracle_workloads"}
    assert _callers(path, {"_oracle_sample", "_oracle_workloads"}) == {"run_ours", "run_reference"}
    # inside run_ours the oracle runs only in the rank-0, single-process CPU-baseline block
    src = open(path, encoding="utf-8").read()
    body = src[src.index("def run_ours("):src.index("def run_reference(")]
    block = body[body.index("if rank == 0 and world == 1 and not args.no_cpu:"):]
    assert body.count("_oracle_sample(") == block.count("_oracle_sample(") == 1
    assert body.count("_oracle_workloads(") == block.count("_oracle_workloads(") == 1


def test_entry_point_uses_the_oracle_only_in_build_and_smoke():
    path = os.path.join(ROOT, "__graft_entry__.py")
    owners = {o for o, _ in _oracle_imports(path)}
    assert owners <= {"build", "smoke", "_smoke_bf16"} and "build" in owners and "smoke" in owners
    assert _callers(path, {"_smoke_bf16"}) == {"smoke"}


def test_binding_raises_without_the_library(tmp_path, monkeypatch):
    monkeypatch.setattr(kda, "_SO", str(tmp_path / "libkda.so"))
    monkeypatch.setattr(kda, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        kda.kda_record_bytes(128, kda.KDA_BF16)
    with pytest.raises(RuntimeError, match="not built"):
        kda.kda_ckpt_positions(0, 1024, 512, 1, False)
