"""The oracle and the CUDA path share no code (static checks on the CPU).

* Nothing in the package (Python binding, layer, build script, CUDA sources
  and headers) or in include/ imports, includes or loads anything of the
  oracle's.
* The oracle imports nothing of the package and includes no CUDA source.
* ``attn_inputs``, the one module both sides use, imports neither.
* ``bench.py`` loads the oracle only inside its CPU-baseline and
  reference-arm functions, never at module level.
* The Python side of the path (binding and layer) holds no attention
  arithmetic and no library or compiler route to one, so nothing can fall
  back from the kernels silently.
"""
from __future__ import annotations

import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "exact_attention_forward_10_gb300")

# functions of bench.py allowed to import the oracle
# the oracle leg of bench.py: the timed sample (self-attention and cache) and
# the per-configuration comparison it runs after that sample
BENCH_ORACLE_USERS = {"cpu_oracle_run", "kv_oracle_run", "per_config_parity"}


def _files(top, exts):
    for d, dirs, fs in os.walk(top):
        dirs[:] = [x for x in dirs if not x.startswith(("_build", "__pycache__"))]
        for f in fs:
            if f.endswith(exts):
                yield os.path.join(d, f)


def _python_imports(path):
    tree = ast.parse(open(path).read())
    out = []
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            out += [a.name.split(".")[0] for a in node.names]
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            out.append(node.module.split(".")[0])
    return out


def test_product_never_touches_the_oracle():
    for path in _files(PKG, (".py",)):
        assert "oracle" not in _python_imports(path), path
        assert "liboracle" not in open(path).read(), path
    for path in list(_files(os.path.join(PKG, "csrc"), (".cu", ".cuh", ".h"))) + \
            list(_files(os.path.join(ROOT, "include"), (".h",))):
        text = open(path).read()
        for inc in re.findall(r'#include\s+[<"]([^>"]+)[>"]', text):
            assert "oracle" not in inc, (path, inc)
        assert "attn_oracle" not in text and "liboracle" not in text, path


def test_oracle_never_touches_the_product():
    for path in _files(os.path.join(ROOT, "oracle"), (".py",)):
        imps = _python_imports(path)
        assert "exact_attention_forward_10_gb300" not in imps, path
        assert "torch" not in imps, path
    for path in _files(os.path.join(ROOT, "oracle"), (".c", ".h")):
        text = open(path).read()
        for inc in re.findall(r'#include\s+[<"]([^>"]+)[>"]', text):
            assert not inc.startswith(("fattn", "ptx", "cuda")), (path, inc)


def test_shared_input_module_imports_neither_side():
    for path in _files(os.path.join(ROOT, "attn_inputs"), (".py",)):
        imps = _python_imports(path)
        assert "oracle" not in imps and "exact_attention_forward_10_gb300" not in imps, path


def test_bench_loads_the_oracle_only_in_its_baseline_functions():
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    users = set()

    def visit(node, func):
        for child in ast.iter_child_nodes(node):
            f = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else func
            if isinstance(child, ast.Import) and any(a.name.split(".")[0] == "oracle"
                                                     for a in child.names):
                users.add(func)
            if isinstance(child, ast.ImportFrom) and (child.module or "").split(".")[0] == "oracle":
                users.add(func)
            visit(child, f)

    visit(tree, None)
    assert None not in users, "bench.py imports the oracle at module level"
    assert users <= BENCH_ORACLE_USERS, users


FORBIDDEN_ON_PATH = ("softmax", "scaled_dot_product_attention", "einsum", "matmul",
                     "bmm", "logsumexp", "torch.exp", "np.exp", "triton", "torch.compile")


def test_python_side_of_the_path_computes_no_attention():
    """The binding and the layer marshal arguments and run the projections
    (``nn.Linear``); every step of the attention itself runs in the CUDA
    kernels, so none of these appear there (no silent host or library
    fallback)."""
    for path in _files(PKG, (".py",)):
        if os.path.basename(path) == "build.py":
            continue
        tree = ast.parse(open(path).read())
        # docstrings (and comments, which the parser drops) may name these
        # things; the code itself may not
        for node in ast.walk(tree):
            body = getattr(node, "body", None)
            if (isinstance(body, list) and body and isinstance(body[0], ast.Expr)
                    and isinstance(body[0].value, ast.Constant)
                    and isinstance(body[0].value.value, str)):
                node.body = body[1:] or [ast.Pass()]
        code = ast.unparse(tree)
        for word in FORBIDDEN_ON_PATH:
            assert word not in code, (path, word)
        assert " @ " not in code, (path, "matrix product")
