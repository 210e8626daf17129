"""The product path has no fallback: the Python package and the CUDA sources
never reach the oracle, and without the built library every call raises."""

import ast
import glob
import os
import re

import pytest

import paged_decode_attention_fp8_gb300 as fm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "paged_decode_attention_fp8_gb300")


def test_package_never_imports_the_oracle():
    for path in glob.glob(os.path.join(PKG, "*.py")):
        tree = ast.parse(open(path).read())
        for node in ast.walk(tree):
            if isinstance(node, ast.Import):
                names = [a.name for a in node.names]
            elif isinstance(node, ast.ImportFrom):
                names = [node.module or ""]
            else:
                continue
            assert not any(n == "oracle" or n.startswith("oracle.") for n in names), path


def test_cuda_sources_never_name_the_oracle():
    for path in glob.glob(os.path.join(PKG, "csrc", "*")) + glob.glob(os.path.join(ROOT, "include", "*.h")):
        assert not re.search(r"\boracle\b", open(path).read()), path


def test_missing_library_raises(monkeypatch):
    monkeypatch.setattr(fm, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libfp8mla.so"))
    monkeypatch.setattr(fm, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        fm.lib()
    with pytest.raises(RuntimeError):
        fm.workspace_bytes(64, 2, 64, 76)
