"""The product path and the oracle share no code.

The package (CUDA sources, host layer, binding) never imports, links or
reads anything under oracle/; the oracle includes nothing from the package
or include/.  The only module both sides' callers use is workloads.py, which
draws numbers and holds none of the collective's arithmetic."""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "allgather_rr_allreduce_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _files(top, exts):
    for d, _, names in os.walk(top):
        if "__pycache__" in d:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def test_package_never_names_the_oracle():
    for f in _files(PKG, (".py", ".cu", ".cuh", ".h", ".cpp")):
        text = open(f).read()
        assert not re.search(r"\boracle\b", text), f"{f} mentions the oracle"


def test_oracle_includes_nothing_from_the_cuda_side():
    for f in _files(ORACLE, (".c", ".py", ".h")):
        text = open(f).read()
        assert "allgather_rr_allreduce_gb300" not in text, f
        assert not re.search(r'#include\s+"', text), f"{f} includes a local header"
        assert "rr.h" not in text and "csrc" not in text, f


def test_workloads_holds_no_collective_arithmetic():
    import ast
    tree = ast.parse(open(os.path.join(ROOT, "workloads.py")).read())
    imported, called = set(), set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            imported |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom):
            imported.add((node.module or "").split(".")[0])
        elif isinstance(node, ast.Call):
            f = node.func
            called.add(f.attr if isinstance(f, ast.Attribute) else getattr(f, "id", ""))
    assert "oracle" not in imported and "allgather_rr_allreduce_gb300" not in imported
    # no summation over ranks
    assert not called & {"sum", "add", "cumsum", "reduce"}, called
