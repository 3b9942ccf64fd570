"""The product path never touches the oracle and has no CPU fallback.

The package's sources are scanned for any import of `oracle`, and loading the
binding against a missing library must raise instead of falling back.
"""
import ast
import importlib.util
import pathlib

import pytest

PKG = pathlib.Path(__file__).resolve().parent.parent / "causal_head_attention_fwd_gb300"


def test_package_never_imports_the_oracle():
    for f in PKG.rglob("*.py"):
        tree = ast.parse(f.read_text())
        for node in ast.walk(tree):
            if isinstance(node, ast.Import):
                assert all(not a.name.split(".")[0] == "oracle" for a in node.names), f
            if isinstance(node, ast.ImportFrom):
                assert (node.module or "").split(".")[0] != "oracle", f


def test_binding_raises_without_the_library(tmp_path):
    # load a private copy of api.py whose library path points at nothing
    src = (PKG / "api.py").read_text()
    fake = tmp_path / "api_copy.py"
    fake.write_text(src.replace('_LIB_PATH = pathlib.Path(__file__).resolve().parent / "libattn.so"',
                                '_LIB_PATH = pathlib.Path(__file__).resolve().parent / "missing_libattn.so"'))
    assert "missing_libattn.so" in fake.read_text()
    spec = importlib.util.spec_from_file_location("api_copy", fake)
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)
