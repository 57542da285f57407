"""The product path has no CPU or oracle fallback.

The package's sources import nothing from the oracle, and asking for the
library when its shared object is missing raises instead of running anything
else.  (The oracle is test infrastructure: only the tests, the package's
smoke check and the benchmark's CPU legs load it.)
"""
import ast
import os

import pytest

import quantized_routed_expert_router_gb300 as moe
from quantized_routed_expert_router_gb300 import _build

PKG = os.path.dirname(os.path.abspath(moe.__file__))


def _imports(path):
    tree = ast.parse(open(path).read(), path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name
        elif isinstance(node, ast.ImportFrom):
            yield node.module or ""


def test_package_never_imports_the_oracle():
    sources = [f for f in os.listdir(PKG) if f.endswith(".py")]
    assert sources
    for f in sources:
        for name in _imports(os.path.join(PKG, f)):
            assert not name.split(".")[0] == "oracle", f"{f} imports {name}"


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(_build, "SO", str(tmp_path / "absent.so"))
    monkeypatch.setattr(moe, "_lib_handle", None)
    with pytest.raises(RuntimeError, match="not built"):
        moe.lib()
