"""The product path has no fallback and the oracle stays apart from it.

- The binding refuses to import when libbi.so is missing (no CPU or PyTorch
  path takes over).
- No module of the product package imports the oracle, and the oracle
  imports nothing of the product package; neither side's C/CUDA sources
  include the other's headers.
"""
import ast
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "invariant_fixed_order_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _py_files(folder):
    for dirpath, _, files in os.walk(folder):
        if "_build" in dirpath or "__pycache__" in dirpath:
            continue
        for f in files:
            if f.endswith(".py"):
                yield os.path.join(dirpath, f)


def _imported_modules(path):
    tree = ast.parse(open(path).read(), path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name
        elif isinstance(node, ast.ImportFrom) and node.level == 0 and node.module:
            yield node.module


def test_binding_refuses_to_import_without_the_library():
    code = ("import invariant_fixed_order_gb300.build as b\n"
            "b.LIB = '/nonexistent/libbi.so'\n"
            "import invariant_fixed_order_gb300.bi\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "not built" in r.stderr


def test_product_package_never_imports_the_oracle():
    files = list(_py_files(PKG))
    assert files
    for path in files:
        for mod in _imported_modules(path):
            assert mod.split(".")[0] != "oracle", f"{path} imports {mod}"


def test_oracle_never_imports_the_product_package():
    for path in _py_files(ORACLE):
        for mod in _imported_modules(path):
            assert mod.split(".")[0] != "invariant_fixed_order_gb300", f"{path} imports {mod}"


def test_c_sources_include_nothing_of_the_other_side():
    inc = re.compile(r'^\s*#\s*include\s*[<"]([^>"]+)[>"]', re.M)
    csrc = os.path.join(PKG, "csrc")
    for f in os.listdir(csrc):
        if f.endswith((".cu", ".cuh", ".h", ".cpp")):
            for h in inc.findall(open(os.path.join(csrc, f)).read()):
                assert "oracle" not in h, f"{f} includes {h}"
    for f in os.listdir(ORACLE):
        if f.endswith((".c", ".h")):
            for h in inc.findall(open(os.path.join(ORACLE, f)).read()):
                assert "bi.h" not in h and "csrc" not in h and "include/" not in h, f"{f} includes {h}"
