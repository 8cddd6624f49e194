"""The oracle and the CUDA path share no code: the oracle's C sources
include only C library headers, no file of the package or its kernels
mentions or imports the oracle, and outside the tests only the build and
smoke entry points and the benchmark's CPU legs load it.  CPU only."""
import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "moe_deferred_finalize_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _files(top, exts):
    for d, _, names in os.walk(top):
        if "_build" in d or "__pycache__" in d:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def test_oracle_c_includes_only_the_c_library():
    allowed = {"math.h", "stdint.h", "string.h", "stdlib.h", "stddef.h"}
    for path in _files(ORACLE, (".c", ".h")):
        for inc in re.findall(r'#\s*include\s*([<"][^>"]+[>"])', open(path).read()):
            assert inc[0] == "<" and inc[1:-1] in allowed, (path, inc)


def test_package_never_refers_to_the_oracle():
    for path in _files(PKG, (".py", ".cu", ".cuh", ".c", ".h")):
        text = open(path).read()
        if path.endswith(".py"):
            for node in ast.walk(ast.parse(text)):
                if isinstance(node, ast.Import):
                    assert not any(a.name.split(".")[0] == "oracle" for a in node.names), path
                if isinstance(node, ast.ImportFrom):
                    assert (node.module or "").split(".")[0] != "oracle", path
        else:
            assert "oracle" not in text and "oref_" not in text, path


def test_only_the_permitted_entry_points_load_the_oracle():
    """Outside tests/: __graft_entry__ (build and smoke) and bench.py's CPU
    legs (the finalize and the all-reduce-fused finalize timed on the host),
    each importing it inside the function that needs it."""
    for name in ("bench.py", "__graft_entry__.py"):
        tree = ast.parse(open(os.path.join(ROOT, name)).read())
        for node in tree.body:       # no module-level import
            if isinstance(node, ast.Import):
                assert not any(a.name.split(".")[0] == "oracle" for a in node.names), name
            if isinstance(node, ast.ImportFrom):
                assert (node.module or "").split(".")[0] != "oracle", name
        users = set()
        for fn in ast.walk(tree):
            if isinstance(fn, ast.FunctionDef):
                for node in ast.walk(fn):
                    mods = [a.name for a in node.names] if isinstance(node, ast.Import) else \
                        [node.module or ""] if isinstance(node, ast.ImportFrom) else []
                    if any(m.split(".")[0] == "oracle" for m in mods):
                        users.add(fn.name)
        allowed = {"bench.py": {"oracle_gbps", "oracle_times", "oracle_allreduce_seconds"},
                   "__graft_entry__.py": {"build", "smoke"}}[name]
        assert users and users <= allowed, (name, users)


def test_no_triton_no_compile_no_cpu_compute_in_the_product():
    """The product (package, kernels, bench, entry points) uses no Triton
    and no torch.compile, and the binding has no compute of its own: it only
    checks, allocates and calls the library."""
    product = list(_files(PKG, (".py", ".cu", ".cuh", ".c"))) + \
        [os.path.join(ROOT, n) for n in ("bench.py", "__graft_entry__.py")]
    for path in product:
        text = open(path).read()
        assert not re.search(r"^\s*(import|from)\s+triton", text, re.M), path
        assert "torch.compile" not in text, path
    binding = open(os.path.join(PKG, "_abi.py")).read()
    for op in ("torch.matmul", "torch.einsum", "index_select", "torch.rsqrt", "rms_norm",
               ".sum(", ".mean(", "torch.topk", "torch.sigmoid", "torch.softmax"):
        assert op not in binding, op
