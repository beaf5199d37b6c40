"""The C-ABI library loads and exports every entry point include/*.h declares (CPU)."""

import ctypes
import glob
import os
import re

import quantized_moe_noaux_b300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(moe_\w+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported():
    declared = declared_functions()
    assert {"moe_layer_create", "moe_layer_forward", "moe_layer_destroy"} <= declared
    lib = ctypes.CDLL(moe.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert declared == set(moe.SYMBOLS), declared ^ set(moe.SYMBOLS)


def test_status_strings_and_null_safety():
    for code, name in moe.STATUS.items():
        assert moe.lib.moe_status_string(code).decode() == name
    moe.lib.moe_layer_destroy(None)                       # NULL is a no-op
    assert moe.lib.moe_layer_forward(None, None, 1, None, None) == 1
    assert moe.lib.moe_layer_status(None) == 1
    assert moe.lib.moe_layer_set_path(None, 0) == 1
    assert moe.lib.moe_layer_create(None, None, None, None) == 1
