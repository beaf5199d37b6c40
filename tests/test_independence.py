"""The oracle and the CUDA path share no code (CPU): no module of the library package or
of the input generator imports the oracle or the tests; the oracle imports neither the
library, the generator, the tests nor ctypes (it never loads the library); no C/CUDA
source includes anything from the oracle or the tests."""

import ast
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def imported_modules(path):
    tree = ast.parse(open(path).read(), filename=path)
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names.update(alias.name.split(".")[0] for alias in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            names.add(node.module.split(".")[0])
    return names


def py_files(*dirs):
    return [p for d in dirs for p in glob.glob(os.path.join(ROOT, d, "**", "*.py"), recursive=True)]


def test_library_and_generator_do_not_import_the_oracle():
    files = py_files("quantized_moe_noaux_b300", "synth")
    assert files
    for path in files:
        bad = imported_modules(path) & {"oracle", "tests"}
        assert not bad, (os.path.relpath(path, ROOT), bad)


def test_oracle_imports_no_product_code():
    files = py_files("oracle")
    assert files
    for path in files:
        bad = imported_modules(path) & {"quantized_moe_noaux_b300", "synth", "tests", "bench", "ctypes"}
        assert not bad, (os.path.relpath(path, ROOT), bad)


def test_cuda_sources_include_nothing_from_oracle_or_tests():
    srcs = [p for ext in ("cu", "cuh", "h") for p in
            glob.glob(os.path.join(ROOT, "quantized_moe_noaux_b300", "csrc", f"*.{ext}"))]
    srcs += glob.glob(os.path.join(ROOT, "include", "*.h"))
    assert srcs
    for path in srcs:
        for inc in re.findall(r'#include\s+[<"]([^>"]+)[>"]', open(path).read()):
            assert "oracle" not in inc and "tests" not in inc, (os.path.relpath(path, ROOT), inc)
