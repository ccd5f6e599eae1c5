"""The library, the binding and the oracle stay independent (CPU only).

* No module of the package (the binding) imports the oracle or the input
  generator, and no oracle module imports the package: the two sides of every
  parity test share nothing but the seeded inputs.
* No CUDA source of the library includes anything outside its own csrc/.
* Importing the binding without libgq.so fails at once (there is no CPU
  fallback): checked on a copy of the package's Python files in a temporary
  directory, so the built library is never touched.
"""
import ast
import os
import re
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "post_weight_quantization_30_b300")
ORACLE = os.path.join(ROOT, "oracle")


def _imported_modules(path):
    tree = ast.parse(open(path, encoding="utf-8").read(), filename=path)
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.level == 0 and node.module:
            names.add(node.module.split(".")[0])
    return names


def _py_files(top):
    for d, _, files in os.walk(top):
        if "__pycache__" in d or "_build" in d:
            continue
        for f in files:
            if f.endswith(".py"):
                yield os.path.join(d, f)


def test_binding_imports_neither_oracle_nor_generator():
    files = list(_py_files(PKG))
    assert files
    for f in files:
        bad = _imported_modules(f) & {"oracle", "synthetic", "numpy", "scipy"}
        assert not bad, f"{os.path.relpath(f, ROOT)} imports {sorted(bad)}"


def test_oracle_does_not_import_the_library():
    files = list(_py_files(ORACLE))
    assert files
    for f in files:
        bad = _imported_modules(f) & {"post_weight_quantization_30_b300", "torch", "ctypes"}
        assert not bad, f"{os.path.relpath(f, ROOT)} imports {sorted(bad)}"


def test_cuda_sources_include_only_their_own_headers():
    csrc = os.path.join(PKG, "csrc")
    sources = [f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h"))]
    assert sources
    for f in sources:
        for inc in re.findall(r'#include\s+"([^"]+)"', open(os.path.join(csrc, f), encoding="utf-8").read()):
            target = os.path.normpath(os.path.join(csrc, inc))
            assert os.path.dirname(target) == csrc or target == os.path.join(ROOT, "include", "gq.h"), (f, inc)


def test_binding_without_library_fails_at_import(tmp_path):
    dst = tmp_path / "post_weight_quantization_30_b300"
    dst.mkdir()
    for f in os.listdir(PKG):
        if f.endswith(".py"):
            shutil.copy(os.path.join(PKG, f), dst / f)
    code = "import post_weight_quantization_30_b300"
    p = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, PYTHONPATH=str(tmp_path)))
    assert p.returncode != 0
    assert "ImportError" in p.stderr and "libgq.so is missing" in p.stderr, p.stderr[-2000:]
