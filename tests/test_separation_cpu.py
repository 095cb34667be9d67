"""The oracle and the CUDA path stay separate (static checks, no GPU).

The oracle is test infrastructure: the product package and its CUDA sources
never import or include it, the oracle imports nothing from the product, and
the only other places that reach it are the bench's CPU-baseline and
reference-arm functions and the smoke check.
"""

import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "tiled_attention_tmem_gb300")


def _imports(path):
    """(module name, enclosing top-level function or None) for every import in a file."""
    tree = ast.parse(open(path, encoding="utf-8").read(), filename=path)
    out = []

    def visit(node, func):
        for child in ast.iter_child_nodes(node):
            f = func
            if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) and func is None:
                f = child.name
            if isinstance(child, ast.Import):
                out.extend((a.name, f) for a in child.names)
            elif isinstance(child, ast.ImportFrom):
                out.append(((child.module or ""), f) if child.level == 0 else ("." + (child.module or ""), f))
            visit(child, f)

    visit(tree, None)
    return out


def _py_files(folder):
    for dirpath, _, files in os.walk(folder):
        for f in files:
            if f.endswith(".py"):
                yield os.path.join(dirpath, f)


def test_product_package_never_imports_the_oracle():
    for path in _py_files(PKG):
        for mod, _ in _imports(path):
            assert not mod.split(".")[0] == "oracle", f"{path} imports {mod}"


def test_cuda_sources_include_nothing_from_the_oracle():
    for folder in (os.path.join(PKG, "csrc"), os.path.join(ROOT, "include")):
        for f in os.listdir(folder):
            text = open(os.path.join(folder, f), encoding="utf-8").read()
            for inc in re.findall(r'#include\s*[<"]([^>"]+)[>"]', text):
                assert "oracle" not in inc, f"{f} includes {inc}"


def test_oracle_imports_only_numpy_and_itself():
    for path in _py_files(os.path.join(ROOT, "oracle")):
        for mod, _ in _imports(path):
            top = mod.split(".")[0]
            assert mod.startswith(".") or top in ("numpy", "__future__"), f"{path} imports {mod}"


def test_oracle_reached_only_from_the_baseline_reference_and_smoke():
    allowed = {
        os.path.join(ROOT, "bench.py"): {"time_oracle", "run_reference"},
        os.path.join(ROOT, "__graft_entry__.py"): {"smoke"},
    }
    for path, funcs in allowed.items():
        users = {f for mod, f in _imports(path) if mod.split(".")[0] == "oracle"}
        assert users and users <= funcs, f"{path}: oracle imported in {users}"


def test_input_module_holds_no_attention_arithmetic():
    """The seeded input generators, shared by both sides, draw and round numbers only:
    no matrix product, exponential, logarithm, maximum or reduction over a tensor."""
    path = os.path.join(PKG, "inputs.py")
    tree = ast.parse(open(path, encoding="utf-8").read())
    banned_calls = {"exp", "exp2", "log", "log2", "max", "maximum", "sum", "matmul", "dot", "einsum",
                    "tensordot", "softmax", "logsumexp", "amax", "cumsum"}
    for node in ast.walk(tree):
        assert not (isinstance(node, ast.BinOp) and isinstance(node.op, ast.MatMult)), "matrix product"
        if isinstance(node, ast.Call):
            fn = node.func
            name = fn.attr if isinstance(fn, ast.Attribute) else getattr(fn, "id", "")
            assert name not in banned_calls, f"inputs.py calls {name}"
