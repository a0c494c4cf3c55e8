"""The product path never reaches the oracle: importing the package loads no
oracle module, and no source of the package (binding, build script, CUDA
and C++ sources, public header) imports, includes or links anything of it.
Only tests, smoke() and the bench's CPU legs may use the oracle."""
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def built():
    import __graft_entry__
    __graft_entry__.build()


def test_importing_the_package_loads_no_oracle_module(built):
    code = ("import sys, adaln_modulate_gb300\n"
            "bad = [m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')]\n"
            "assert not bad, bad\n")
    subprocess.run([sys.executable, "-c", code], cwd=ROOT, check=True)


def test_product_sources_do_not_refer_to_the_oracle():
    pkg = os.path.join(ROOT, "adaln_modulate_gb300")
    files = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))]
    for d, _, names in os.walk(pkg):
        if "_build" in d or "__pycache__" in d:
            continue
        files += [os.path.join(d, n) for n in names if n.endswith((".py", ".cu", ".cuh", ".h", ".cpp"))]
    assert files
    pattern = re.compile(r"^\s*(import\s+oracle|from\s+oracle|#\s*include\s*[<\"][^>\"]*oracle)|liboracle|oracle/",
                         re.M)
    hits = [f for f in files if pattern.search(open(f, encoding="utf-8").read())]
    assert not hits, hits
