"""The product path and the oracle stay apart (CPU only).

The CUDA library and its Python binding never import, include or call the
oracle, the oracle never touches the product path, and the binding refuses to
run without its compiled library instead of falling back to anything else.
"""
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "sparse_kv_cache_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _sources(top, exts):
    for d, _, files in os.walk(top):
        if "_build" in d or "__pycache__" in d:
            continue
        for f in files:
            if f.endswith(exts):
                yield os.path.join(d, f)


def test_product_sources_never_name_the_oracle():
    pat = re.compile(r"\boracle\b|shadowkv_ref")
    hits = [p for p in _sources(PKG, (".py", ".cu", ".cuh", ".h", ".cpp")) if pat.search(open(p).read())]
    hits += [p for p in _sources(os.path.join(ROOT, "include"), (".h",)) if pat.search(open(p).read())]
    assert hits == []


def test_oracle_never_touches_the_product_path():
    pat = re.compile(r"sparse_kv_cache_gb300|libshadowkv|ctypes|torch\.cuda")
    assert [p for p in _sources(ORACLE, (".py",)) if pat.search(open(p).read())] == []


def test_importing_the_package_loads_no_oracle_module():
    code = ("import sys; import sparse_kv_cache_gb300 as skv; "
            "print(sorted(m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')))")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, check=True)
    assert out.stdout.strip() == "[]"


def test_binding_refuses_to_run_without_the_library():
    from sparse_kv_cache_gb300 import _binding
    saved = _binding._lib
    _binding._lib = None
    try:
        with pytest.raises(ImportError):
            _binding.load(os.path.join(ROOT, "no_such_dir", "libshadowkv.so"))
    finally:
        _binding._lib = saved
