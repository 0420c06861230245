"""The oracle and the CUDA path share no code: the package never imports or
includes the oracle, the oracle never imports the package or the library,
importing the package does not load the oracle, and bench.py reaches the
oracle only inside its CPU legs (no module-level import)."""
import ast
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "paged_kv_decode_bind_gb300")


def _files(top, exts):
    for d, _, names in os.walk(top):
        if "_build" in d or "__pycache__" in d:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def test_package_does_not_reach_the_oracle():
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle|#\s*include\s*[\"<].*oracle)", re.M)
    for f in _files(PKG, (".py", ".cu", ".cuh", ".h")):
        with open(f) as fh:
            assert not pat.search(fh.read()), f


def test_oracle_does_not_reach_the_package():
    # no import of the package, no loading of a shared library, no path into
    # the kernel sources (its docstrings may name the package)
    for f in _files(os.path.join(ROOT, "oracle"), (".py",)):
        with open(f) as fh:
            src = fh.read()
        for node in ast.walk(ast.parse(src)):
            if isinstance(node, ast.Import):
                assert not any(a.name.startswith(("paged_kv_decode_bind_gb300", "ctypes"))
                               for a in node.names), f
            if isinstance(node, ast.ImportFrom):
                assert not (node.module or "").startswith(("paged_kv_decode_bind_gb300",
                                                           "ctypes")), f
        assert not re.search(r"CDLL|libpkv\.so|csrc/", src), f


def test_importing_the_package_does_not_load_the_oracle():
    code = ("import sys; import paged_kv_decode_bind_gb300; "
            "print(any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules))")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0, out.stderr[-500:]
    assert out.stdout.strip() == "False"


def test_bench_imports_the_oracle_only_inside_functions():
    with open(os.path.join(ROOT, "bench.py")) as fh:
        tree = ast.parse(fh.read())
    for node in tree.body:  # module level only
        if isinstance(node, ast.Import):
            assert not any(a.name.split(".")[0] == "oracle" for a in node.names)
        if isinstance(node, ast.ImportFrom):
            assert (node.module or "").split(".")[0] != "oracle"
