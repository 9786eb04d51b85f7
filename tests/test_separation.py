"""The oracle and the CUDA path share no code: no module of the product
package imports the oracle, no oracle module imports the product, and the
seeded input generators import neither.  Checked on the import statements of
every source file (AST), so a lazy import inside a function counts too."""

import ast
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PRODUCT = "paged_kv_cache_254_gb300"


def imported_roots(path):
    tree = ast.parse(open(path, encoding="utf-8").read(), filename=path)
    roots = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            roots.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.level == 0 and node.module:
            roots.add(node.module.split(".")[0])
    return roots


def py_files(folder):
    for dirpath, _, names in os.walk(os.path.join(ROOT, folder)):
        if "__pycache__" in dirpath:
            continue
        for n in names:
            if n.endswith(".py"):
                yield os.path.join(dirpath, n)


@pytest.mark.parametrize("folder,forbidden", [
    (PRODUCT, {"oracle", "tests"}),
    ("oracle", {PRODUCT, "tests", "bench"}),
    ("workloads", {"oracle", PRODUCT, "tests"}),
])
def test_no_shared_code(folder, forbidden):
    files = list(py_files(folder))
    assert files
    for f in files:
        bad = imported_roots(f) & forbidden
        assert not bad, f"{os.path.relpath(f, ROOT)} imports {sorted(bad)}"


def test_native_sources_do_not_reach_the_oracle():
    # the CUDA/C++ sources include only their own headers and the toolkit's
    csrc = os.path.join(ROOT, PRODUCT, "csrc")
    for n in os.listdir(csrc):
        text = open(os.path.join(csrc, n), encoding="utf-8").read()
        assert "oracle" not in text.lower(), n


def test_bench_uses_the_oracle_only_for_the_cpu_baseline():
    tree = ast.parse(open(os.path.join(ROOT, "bench.py"), encoding="utf-8").read())
    users = set()
    for fn in ast.walk(tree):
        if isinstance(fn, ast.FunctionDef):
            for node in ast.walk(fn):
                if isinstance(node, ast.ImportFrom) and node.module and node.module.split(".")[0] == "oracle":
                    users.add(fn.name)
    assert users == {"cpu_worker"}
    assert "oracle" not in {a.name.split(".")[0] for node in tree.body if isinstance(node, ast.Import)
                            for a in node.names}
