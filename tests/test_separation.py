"""The CUDA path and the oracle share nothing (CPU).

The product package neither imports the oracle nor reads its sources, the
two sides include no common header, and the product library exports none of
the oracle's symbols; the only module both use is synth.py, which draws
random numbers and holds none of the method's arithmetic."""
import ast
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "w4a16_decode_paged_gb300")


def _imports(path):
    tree = ast.parse(open(path).read(), path)
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            names.add(node.module.split(".")[0])
    return names


def test_product_python_never_imports_the_oracle():
    for path in glob.glob(os.path.join(PKG, "*.py")):
        assert "oracle" not in _imports(path), path


def test_synth_holds_no_method_arithmetic():
    imports = _imports(os.path.join(PKG, "synth.py"))
    assert imports <= {"__future__", "numpy"}, imports


def test_cuda_sources_and_oracle_share_no_include():
    csrc = glob.glob(os.path.join(PKG, "csrc", "*"))
    local = set()
    for path in csrc:
        local |= set(re.findall(r'#include\s+"([^"]+)"', open(path).read()))
    assert local <= {os.path.basename(p) for p in csrc} | {"w4a16.h"}, local   # its own headers and the ABI
    oracle_inc = set(re.findall(r'#include\s+[<"]([^>"]+)[>"]', open(os.path.join(ROOT, "oracle", "oracle.c")).read()))
    assert not oracle_inc & {os.path.basename(p) for p in csrc}
    assert oracle_inc <= {"math.h", "stdint.h", "stdlib.h", "string.h", "omp.h"}, oracle_inc
    for path in csrc:
        assert "oracle" not in open(path).read().lower(), path


def test_library_exports_no_oracle_symbol():
    from w4a16_decode_paged_gb300 import build
    so = build.build()
    nm = subprocess.run(["nm", "-D", "--defined-only", so], capture_output=True, text=True)
    if nm.returncode != 0:
        pytest.skip("nm unavailable")
    syms = {line.split()[-1] for line in nm.stdout.splitlines() if line.strip()}
    assert not {s for s in syms if s.startswith("orc_")}
