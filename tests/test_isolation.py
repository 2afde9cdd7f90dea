"""The oracle and the CUDA path share nothing, and the product path has no
CPU fallback (no GPU needed).

* No module of the package imports the oracle, and no CUDA or C source of the
  package includes an oracle header; the oracle's C source includes nothing
  of the package.
* Importing the package does not load the oracle.
* On a machine without a GPU, creating a context raises instead of computing
  anything on the CPU."""
import ast
import glob
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "combine_get_dispatch_histograms_gb300")


def _imports(path):
    tree = ast.parse(open(path).read())
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            names.add(node.module.split(".")[0])
    return names


def test_package_never_imports_the_oracle():
    files = glob.glob(os.path.join(PKG, "**", "*.py"), recursive=True)
    assert files
    for f in files:
        assert "oracle" not in _imports(f), f
    for f in glob.glob(os.path.join(ROOT, "include", "*.h")) + glob.glob(os.path.join(PKG, "csrc", "*")):
        src = open(f).read()
        assert not re.search(r"#\s*include\s*[<\"][^>\"]*oracle", src), f
        assert "orc_" not in src, f


def test_oracle_includes_nothing_of_the_package():
    for f in glob.glob(os.path.join(ROOT, "oracle", "*.[ch]")):
        for inc in re.findall(r"#\s*include\s*[<\"]([^>\"]+)[>\"]", open(f).read()):
            assert inc in ("ep_oracle.h", "stdint.h", "stddef.h", "stdlib.h", "string.h", "math.h",
                           "stdio.h"), (f, inc)
    for f in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        assert "combine_get_dispatch_histograms_gb300" not in _imports(f), f


def test_importing_the_package_does_not_load_the_oracle():
    code = ("import sys; import combine_get_dispatch_histograms_gb300 as p; "
            "import combine_get_dispatch_histograms_gb300.buffer, combine_get_dispatch_histograms_gb300.dist; "
            "assert 'oracle' not in sys.modules, sorted(m for m in sys.modules if 'oracle' in m)")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_no_cpu_fallback_without_a_gpu():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from combine_get_dispatch_histograms_gb300 import Context, LLBuffer
    with pytest.raises(RuntimeError):
        Context(4, 8, 2, 16, 128)
    with pytest.raises(RuntimeError):
        LLBuffer(4, 8, 2, 16, 128, 16)
