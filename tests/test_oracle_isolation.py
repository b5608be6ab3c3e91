"""The oracle is test infrastructure: the product path never reaches it,
and it has no fallback of any kind.

Static and import-time checks, no GPU: the package's sources never name the
oracle, importing the package loads no oracle module, and the only places
outside tests/ that import it are the bench's CPU baseline and reference
arm and the smoke check.  Without an up-to-date libvr.so every entry point
raises.
"""

import ast
import os
import subprocess
import sys

import pytest

from tests.conftest import ROOT

PACKAGE = os.path.join(ROOT, "double_binary_tree_gb300")
ALLOWED = {
    # the CPU baseline and the reference arm, and the worker task both spread
    # over the host's cores
    "bench.py": {"cpu_baseline", "reference_arm", "_oracle_channel"},
    "__graft_entry__.py": {"smoke"},
}


def _package_sources():
    for dirpath, dirnames, filenames in os.walk(PACKAGE):
        dirnames[:] = [d for d in dirnames if not d.startswith(("_build", "__pycache__"))]
        for f in filenames:
            if f.endswith((".py", ".cc", ".cu", ".cuh", ".h")):
                yield os.path.join(dirpath, f)


def test_package_sources_never_name_the_oracle():
    files = list(_package_sources())
    assert any(f.endswith("api.cc") for f in files)
    for path in files:
        with open(path, encoding="utf-8") as fh:
            assert "oracle" not in fh.read(), path


def test_importing_the_package_loads_no_oracle_module():
    code = ("import sys; import double_binary_tree_gb300; "
            "print(sorted(m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')))")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "[]"


def _oracle_imports(tree):
    """(enclosing top-level function or None, line) of every import of the
    oracle package in a module's syntax tree."""
    found = []

    def visit(node, fn):
        for child in ast.iter_child_nodes(node):
            here = child.name if isinstance(child, ast.FunctionDef) and fn is None else fn
            if isinstance(child, ast.Import):
                for a in child.names:
                    if a.name == "oracle" or a.name.startswith("oracle."):
                        found.append((fn, child.lineno))
            elif isinstance(child, ast.ImportFrom):
                if child.module and (child.module == "oracle" or child.module.startswith("oracle.")):
                    found.append((fn, child.lineno))
            visit(child, here)

    visit(tree, None)
    return found


def test_oracle_imported_only_where_allowed():
    for name, allowed in ALLOWED.items():
        with open(os.path.join(ROOT, name), encoding="utf-8") as fh:
            tree = ast.parse(fh.read())
        sites = _oracle_imports(tree)
        assert sites, name
        for fn, line in sites:
            assert fn in allowed, "%s:%d imports the oracle in %s" % (name, line, fn)
    with open(os.path.join(ROOT, "workloads.py"), encoding="utf-8") as fh:
        assert not _oracle_imports(ast.parse(fh.read()))


# ------------------------------------------------------------ no fallback
def test_missing_library_raises(monkeypatch):
    """Without libvr.so every entry point raises: there is no other path."""
    import double_binary_tree_gb300 as vr
    monkeypatch.setattr(vr, "_lib", None)
    monkeypatch.setattr(vr, "LIB", os.path.join(ROOT, "no_such_dir", "libvr.so"))
    with pytest.raises(ImportError, match="not built"):
        vr.vr_build_ring(4, 2)
    with pytest.raises(ImportError, match="not built"):
        vr.vr_get_error_string(0)


def test_stale_library_raises(monkeypatch):
    """A library older than its sources (or built elsewhere) is not loaded."""
    import double_binary_tree_gb300 as vr
    monkeypatch.setattr(vr, "_lib", None)
    monkeypatch.setattr(vr, "is_fresh", lambda debug=False: False)
    with pytest.raises(ImportError, match="older than its sources"):
        vr.vr_build_ring(4, 2)
