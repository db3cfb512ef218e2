"""Structural checks (no GPU): the oracle and the CUDA path share no code, and
the product path has no fallback when its library is missing."""
import ast
import os
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "nvfp4_quantized_matmul_gb300")


def imported_modules(path):
    tree = ast.parse(open(path).read())
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names.update(a.name for a in node.names)
        elif isinstance(node, ast.ImportFrom):
            names.add(node.module or "")
    return names


def test_package_never_imports_the_oracle():
    for f in os.listdir(PKG):
        if f.endswith(".py"):
            mods = imported_modules(os.path.join(PKG, f))
            assert not any(m == "oracle" or m.startswith("oracle.") for m in mods), f


def test_oracle_never_imports_the_package():
    odir = os.path.join(ROOT, "oracle")
    for f in os.listdir(odir):
        if f.endswith(".py"):
            mods = imported_modules(os.path.join(odir, f))
            assert not any("nvfp4_quantized_matmul_gb300" in m for m in mods), f


def test_native_sources_do_not_reach_the_oracle():
    for d in (os.path.join(PKG, "csrc"), os.path.join(ROOT, "include")):
        for f in os.listdir(d):
            text = open(os.path.join(d, f)).read()
            assert "oracle" not in text, f


def test_binding_fails_loudly_without_its_library(tmp_path):
    """A copy of the package without libnvfp4.so cannot be imported for use:
    the binding raises instead of falling back to anything on the host."""
    dst = tmp_path / "nvfp4_quantized_matmul_gb300"
    dst.mkdir()
    for f in ("__init__.py", "binding.py", "synth.py"):
        shutil.copy(os.path.join(PKG, f), dst / f)
    code = "import nvfp4_quantized_matmul_gb300.binding"
    r = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, capture_output=True, text=True,
                       env={**os.environ, "PYTHONPATH": str(tmp_path)})
    assert r.returncode != 0
    assert "libnvfp4.so" in (r.stderr + r.stdout)
