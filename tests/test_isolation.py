"""The oracle and the CUDA path stay apart (no GPU).

The product (the package and its C ABI header) never imports, includes or
loads the oracle, so nothing it computes can come from it; the oracle never
reaches into the product, so its results are independent of the kernels;
and the benchmark and entry module touch the oracle only in their checking
legs: the cpu_baseline leg and the reference arm of bench.py, and smoke()
(build() only compiles it)."""
import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "tiled_tensor_core_gemm_gb300")


def _files(top, exts):
    for d, dirs, names in os.walk(top):
        dirs[:] = [x for x in dirs if not x.startswith(("_build", "__pycache__"))]
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def test_product_never_reaches_the_oracle():
    pat = re.compile(r"^\s*(import\s+oracle\b|from\s+oracle\b)|gemm_oracle|libgemm_oracle|oracle/", re.M)
    files = list(_files(PKG, (".py", ".cu", ".cuh", ".h", ".cpp"))) + list(_files(os.path.join(ROOT, "include"), (".h",)))
    assert files
    hits = [f for f in files if pat.search(open(f).read())]
    assert not hits, hits


def test_oracle_never_reaches_the_product():
    files = list(_files(os.path.join(ROOT, "oracle"), (".py", ".c", ".h")))
    assert any(f.endswith("gemm_oracle.c") for f in files)
    for f in files:
        text = open(f).read()
        assert "tiled_tensor_core_gemm_gb300" not in text and "csrc" not in text, f
        for inc in re.findall(r'^\s*#\s*include\s*(.+)$', text, re.M):
            assert inc.strip().startswith("<"), (f, inc)       # standard headers only


def _oracle_imports_by_function(path):
    """Names of the functions that import the oracle ('<module>' at top level)."""
    tree = ast.parse(open(path).read())
    found = []

    def visit(node, where):
        for child in ast.iter_child_nodes(node):
            inner = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else where
            if isinstance(child, ast.Import) and any(a.name.split(".")[0] == "oracle" for a in child.names):
                found.append(where)
            if isinstance(child, ast.ImportFrom) and (child.module or "").split(".")[0] == "oracle":
                found.append(where)
            visit(child, inner)

    visit(tree, "<module>")
    return found


def test_bench_uses_the_oracle_only_in_its_checking_legs():
    where = _oracle_imports_by_function(os.path.join(ROOT, "bench.py"))
    assert where and set(where) <= {"_time_oracle", "_parity_rows", "run_reference"}, where


def test_entry_module_uses_the_oracle_only_to_build_it_and_in_smoke():
    where = _oracle_imports_by_function(os.path.join(ROOT, "__graft_entry__.py"))
    assert where and set(where) <= {"build", "smoke"}, where
