"""The product path and the CPU oracle share no code: no module of the package
imports the oracle, no CUDA source includes an oracle file, the library is
built from the package's sources alone, and the oracle neither imports the
package nor includes its headers."""
import ast
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "allreduce_residual_rmsnorm_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def files(top, exts):
    for d, _, fs in os.walk(top):
        if "__pycache__" in d:
            continue
        for f in fs:
            if f.endswith(exts):
                yield os.path.join(d, f)


def imported_modules(path):
    tree = ast.parse(open(path).read(), path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name.split(".")[0]
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            yield node.module.split(".")[0]


def includes(path):
    return re.findall(r'^\s*#\s*include\s*[<"]([^>"]+)[>"]', open(path).read(), re.M)


@pytest.mark.parametrize("path", sorted(files(PKG, (".py",))), ids=os.path.basename)
def test_package_modules_do_not_import_the_oracle(path):
    assert "oracle" not in set(imported_modules(path)), path


@pytest.mark.parametrize("path", sorted(files(PKG, (".cu", ".cuh", ".h"))), ids=os.path.basename)
def test_cuda_sources_include_no_oracle_file(path):
    for inc in includes(path):
        assert "oracle" not in inc, (path, inc)


def test_library_is_built_from_package_sources_only():
    from allreduce_residual_rmsnorm_gb300 import build as BUILD
    srcs = BUILD.sources()
    assert srcs and all(os.path.dirname(s) == os.path.join(PKG, "csrc") for s in srcs), srcs


@pytest.mark.parametrize("path", sorted(files(ORACLE, (".py", ".c", ".h"))), ids=os.path.basename)
def test_oracle_uses_nothing_of_the_package(path):
    if path.endswith(".py"):
        mods = set(imported_modules(path))
        assert "allreduce_residual_rmsnorm_gb300" not in mods and "bench" not in mods, path
    else:
        for inc in includes(path):
            assert "ar_fusion" not in inc and "csrc" not in inc and not inc.endswith(".cuh"), \
                (path, inc)
