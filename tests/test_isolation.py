"""The CUDA path and the CPU oracle share no code, and the oracle stays test
infrastructure.

Static checks over the sources: the product package (kernels, ABI, binding)
never names the oracle; the oracle includes and imports nothing of the
product; the seeded input generators import neither; the benchmark touches
the oracle only inside its two CPU legs (the CPU baseline and the
reference arm); no tracked file reads the scratch folder.
"""
import ast
import os
import re
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "hadamard_precision_backprop_gb300")


def _files(top, exts):
    for dirpath, dirnames, filenames in os.walk(top):
        dirnames[:] = [d for d in dirnames if not d.startswith(("_build", "__pycache__"))]
        for fn in filenames:
            if fn.endswith(exts):
                yield os.path.join(dirpath, fn)


def _imports(path):
    tree = ast.parse(open(path).read(), path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name.split(".")[0], node
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            yield node.module.split(".")[0], node


def test_product_never_names_the_oracle():
    srcs = list(_files(PKG, (".py", ".cu", ".cuh", ".h", ".cpp")))
    srcs += list(_files(os.path.join(ROOT, "include"), (".h",)))
    assert srcs
    for path in srcs:
        text = open(path).read()
        assert not re.search(r"\boracle\b|\borc_\w+|hlq_oracle", text), path
        if path.endswith(".py"):
            mods = {m for m, _ in _imports(path)}
            assert not mods & {"oracle", "tests", "workloads", "bench"}, (path, mods)


def test_oracle_includes_and_imports_nothing_of_the_product():
    for path in _files(os.path.join(ROOT, "oracle"), (".c", ".h")):
        for inc in re.findall(r'#include\s*[<"]([^>"]+)[>"]', open(path).read()):
            assert inc in {"math.h", "stddef.h", "stdint.h", "string.h", "stdlib.h",
                           "stdio.h"}, (path, inc)
    for path in _files(os.path.join(ROOT, "oracle"), (".py",)):
        mods = {m for m, _ in _imports(path)}
        assert not mods & {"hadamard_precision_backprop_gb300", "torch", "workloads",
                           "bench", "tests"}, (path, mods)
        assert "hadamard_precision_backprop_gb300" not in open(path).read(), path


def test_input_generators_import_neither_side():
    path = os.path.join(ROOT, "workloads.py")
    mods = {m for m, _ in _imports(path)}
    # scipy.special.erf shapes the exact-erf GELU inputs of one workload
    assert mods <= {"__future__", "dataclasses", "math", "numpy", "scipy"}, mods


def test_bench_runs_the_oracle_only_in_its_cpu_legs():
    path = os.path.join(ROOT, "bench.py")
    tree = ast.parse(open(path).read(), path)
    allowed = {"oracle_layer_seconds"}
    for node in ast.walk(tree):
        if isinstance(node, ast.FunctionDef):
            for sub in ast.walk(node):
                if isinstance(sub, (ast.Import, ast.ImportFrom)):
                    names = ([a.name for a in sub.names] if isinstance(sub, ast.Import)
                             else [sub.module or ""])
                    if any(n.split(".")[0] == "oracle" for n in names):
                        assert node.name in allowed, node.name
    top = [m for m, node in _imports(path) if node in tree.body]
    assert "oracle" not in top
    # the function that runs the oracle is called only by the two CPU legs
    callers = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.FunctionDef):
            for sub in ast.walk(node):
                if (isinstance(sub, ast.Call) and isinstance(sub.func, ast.Name)
                        and sub.func.id == "oracle_layer_seconds"):
                    callers.add(node.name)
    assert callers == {"cpu_baseline", "run_reference"}, callers


def test_no_tracked_file_reads_the_scratch_folder():
    out = subprocess.run(["git", "ls-files"], cwd=ROOT, capture_output=True, text=True)
    if out.returncode != 0:
        return                                     # not a git checkout
    for rel in out.stdout.split():
        if rel.startswith("_work/"):
            raise AssertionError(f"scratch file tracked: {rel}")
        if rel.endswith((".py", ".cu", ".cuh", ".h", ".c", ".sh")):
            if rel == "tests/test_isolation.py":
                continue
            text = open(os.path.join(ROOT, rel)).read()
            assert not re.search(r"(?<!\w)_work\b", text), rel
