"""The oracle stays test infrastructure: the product never reaches it.

Only the tests, the smoke check and bench.py's CPU-baseline legs (and its
reference arm, which times the oracle) may import the oracle.  The package
(binding, harness, CUDA sources) must not import, include or link it, so that
no result of the CUDA path can come from the CPU.
"""

import ast
import glob
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "context_decode_attention_gb300")


def _imports_oracle(node):
    if isinstance(node, ast.Import):
        return any(a.name == "oracle" or a.name.startswith("oracle.") for a in node.names)
    if isinstance(node, ast.ImportFrom):
        return (node.module or "").split(".")[0] == "oracle"
    return False


def test_package_sources_never_name_the_oracle():
    for path in glob.glob(os.path.join(PKG, "**", "*.py"), recursive=True):
        tree = ast.parse(open(path).read())
        assert not any(_imports_oracle(n) for n in ast.walk(tree)), path
    for path in glob.glob(os.path.join(PKG, "csrc", "*")):
        text = open(path).read().lower()
        assert "oracle" not in text and "liboracle" not in text, path


def test_importing_the_package_loads_no_oracle():
    code = ("import sys, context_decode_attention_gb300, context_decode_attention_gb300.harness; "
            "print('oracle' in sys.modules)")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == "False"


def test_bench_reaches_the_oracle_only_in_its_baseline_legs():
    src = open(os.path.join(ROOT, "bench.py")).read()
    tree = ast.parse(src)
    allowed_functions = {"cpu_oracle_sample"}  # the bounded timing sample
    found = 0

    def visit(node, func, guarded):
        nonlocal found
        if isinstance(node, ast.FunctionDef):
            func = node.name
        if isinstance(node, ast.If) and "no_cpu_baseline" in ast.get_source_segment(src, node.test):
            guarded = True
        if _imports_oracle(node):
            found += 1
            assert func in allowed_functions or guarded, f"oracle imported at line {node.lineno} in {func}"
        for child in ast.iter_child_nodes(node):
            visit(child, func, guarded)

    visit(tree, None, False)
    assert found >= 1
    # the reference arm times the oracle through cpu_oracle_sample only
    ref = next(n for n in tree.body if isinstance(n, ast.FunctionDef) and n.name == "run_reference")
    assert not any(_imports_oracle(n) for n in ast.walk(ref))
