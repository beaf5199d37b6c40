"""The C-ABI library loads and exports every entry point include/*.h declares (CPU)."""

import ctypes
import glob
import os
import re

import pytest

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


def _cfg(**over):
    base = dict(hidden=6144, inter=2048, n_experts=256, top_k=8, n_group=8, topk_group=4,
                max_tokens=64, routed_scaling_factor=2.5, weight_format=moe.W_INT4_G32,
                shared_format=moe.W_INT4_G32, act_dtype=moe.DT_BF16, router_dtype=moe.DT_F32)
    base.update(over)
    return moe.Config(**base)


@pytest.mark.parametrize("over,code", [
    (dict(hidden=0), 1), (dict(top_k=0), 1), (dict(max_tokens=0), 1),
    (dict(routed_scaling_factor=0.0), 1), (dict(routed_scaling_factor=float("nan")), 1),
    (dict(weight_format=7), 2), (dict(shared_format=9), 2), (dict(act_dtype=5), 2),
    (dict(router_dtype=5), 2),
    (dict(hidden=6000), 2),                       # H not a multiple of 256
    (dict(inter=2000), 2),                        # I not a multiple of 64
    (dict(n_experts=250), 2),                     # E not a multiple of n_group
    (dict(n_group=64, n_experts=256), 2),         # more than 32 groups
    (dict(n_experts=16, n_group=16), 2),          # one expert per group
    (dict(topk_group=9), 2),                      # more kept groups than groups
    (dict(top_k=33), 2),                          # top_k above the selection limit
    (dict(n_experts=16, n_group=8, topk_group=1, top_k=3), 2),   # top_k > kept experts
    (dict(max_tokens=16385), 2),
    (dict(expert_top_p=float("nan")), 1),          # adaptive top-p NaN
    (dict(weight_format=moe.W_INT8_ROW), 2),       # shared expert neither the routed format nor bf16
    (dict(act_quant=2), 2),                        # unknown activation quantisation
    (dict(act_quant=1, weight_format=moe.W_NVFP4, shared_format=moe.W_NVFP4), 2),   # Q8_0 + NVFP4
    (dict(act_quant=1, weight_format=moe.W_INT4_ROW, shared_format=moe.W_BF16), 2),  # Q8_0, bf16 shared
])
def test_create_rejects_bad_configs_before_touching_the_device(over, code):
    """moe_layer_create checks the configuration first (no CUDA call, so this runs on CPU),
    returns the documented status and leaves *out NULL."""
    cfg = _cfg(**over)
    w = moe.Weights()
    out = ctypes.c_void_p(1)
    rc = moe.lib.moe_layer_create(ctypes.byref(cfg), ctypes.byref(w), None, ctypes.byref(out))
    assert rc == code, (over, rc)
    assert out.value is None


# the limits documented with moe_config, each just inside and just outside
_SMALL = dict(inter=64, n_experts=8, n_group=4, topk_group=2, top_k=4)


@pytest.mark.parametrize("over,accepted", [
    (dict(hidden=14336, **_SMALL), True), (dict(hidden=14592, **_SMALL), False),
    (dict(n_experts=1024, n_group=32), True), (dict(n_experts=1056, n_group=32), False),
    (dict(n_experts=64, n_group=32, topk_group=32, top_k=32), True),
    (dict(n_experts=66, n_group=33, topk_group=32, top_k=8), False),
    (dict(n_experts=64, n_group=8, topk_group=4, top_k=32), True),    # 4 groups of 8 hold 32
    (dict(n_experts=64, n_group=8, topk_group=3, top_k=25), False),   # 3 groups of 8 hold 24
    (dict(max_tokens=16384), True), (dict(max_tokens=16385, top_k=1), False),
    # work list: 8191 * 32 / 4 + 256 + 2048 + 1 = 67,833 > 65535; 7,400 tokens: 61,307
    (dict(n_experts=256, n_group=8, topk_group=8, top_k=32, max_tokens=8191), False),
    (dict(n_experts=256, n_group=8, topk_group=8, top_k=32, max_tokens=7400), True),
])
def test_create_limits_at_their_boundaries(over, accepted):
    """A configuration inside every documented limit passes validation (creation then stops
    at the NULL weights, or at the missing device: MOE_ERR_INVALID_ARG or MOE_ERR_CUDA); one
    step outside a limit is MOE_ERR_UNSUPPORTED."""
    cfg = _cfg(**over)
    w = moe.Weights()
    out = ctypes.c_void_p(1)
    rc = moe.lib.moe_layer_create(ctypes.byref(cfg), ctypes.byref(w), None, ctypes.byref(out))
    assert (rc in (1, 4)) if accepted else (rc == 2), (over, rc)
    assert out.value is None


@pytest.mark.parametrize("over,slots,code", [
    (dict(), 63, 1),                                             # fewer slots than one forward needs (64 * 8 > 256 -> 256)
    (dict(max_tokens=4), 31, 1),                                 # min(E, 4 * 8) = 32
    (dict(max_tokens=4), 257, 1),                                # more slots than experts
    (dict(max_tokens=4, weight_format=moe.W_NVFP4, shared_format=moe.W_NVFP4), 64, 2),   # int4_g32 only
    (dict(max_tokens=4, act_quant=1), 64, 2),
])
def test_create_cached_rejects_before_touching_the_device(over, slots, code):
    cfg = _cfg(**over)
    w = moe.Weights()
    out = ctypes.c_void_p(1)
    rc = moe.lib.moe_layer_create_cached(ctypes.byref(cfg), ctypes.byref(w), slots, None, ctypes.byref(out))
    assert rc == code, (over, slots, rc)
    assert out.value is None


def test_debug_and_test_hooks_reject_bad_arguments():
    """Host-side argument checks of the debug and test hooks (no device work)."""
    assert moe.lib.moe_test_fail_allocation(-1) == 1
    assert moe.lib.moe_test_fail_allocation(0) == 0
    assert moe.lib.moe_check_routing(None, None, None, 4, 2, 8, None, None) == 1
    assert moe.lib.moe_layer_set_debug_checks(None, 1) == 1
    assert moe.lib.moe_layer_set_test_activation(None, 1) == 1
    assert moe.lib.moe_layer_prefetch(None, None, 1, None) == 1
    assert moe.lib.moe_layer_cache_stats(None, None) == 1


# moe_route_noalloc checks every argument before its first CUDA call, so its refusals can
# be exercised with stand-in addresses that are never dereferenced. Where a GPU is visible
# the tests are skipped: stand-in addresses must never be able to reach a kernel launch.
_A = 1 << 20                     # a 16-byte-aligned stand-in address
_NOALLOC = dict(x=_A, act=1, T=4, H=256, rw=_A, rdt=0, bias=_A, E=16, n_group=4, topk_group=2,
                top_k=4, rsf=2.5, ids=_A, w=_A, off=_A, ent=_A)


def _gpu_visible():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.mark.skipif(_gpu_visible(), reason="stand-in addresses: CPU only")
@pytest.mark.parametrize("over,code", [
    (dict(T=-1), 1), (dict(H=0), 1), (dict(E=0), 1), (dict(n_group=0), 1),
    (dict(topk_group=0), 1), (dict(top_k=0), 1), (dict(act=5), 1), (dict(rdt=5), 1),
    (dict(rsf=0.0), 1), (dict(rsf=float("nan")), 1),
    (dict(E=1056, n_group=32), 2),                  # more than 1024 experts
    (dict(E=18), 2),                                # n_group does not divide E
    (dict(E=66, n_group=33), 2),                    # more than 32 groups
    (dict(E=8, n_group=8, topk_group=2), 2),        # one expert per group
    (dict(topk_group=5), 2),                        # more kept groups than groups
    (dict(topk_group=2, top_k=9), 2),               # 2 kept groups of 4 hold 8
    (dict(E=256, n_group=8, topk_group=8, top_k=33), 2),
    (dict(T=257, E=1024, n_group=32), 2),           # T * E = 263168 logits > 262144
    (dict(T=256, E=1024, n_group=32), 4),           # 262144: accepted (then no device)
    # work list: T * k / 4 + min(T * k, E) + 1 = 8193 > 8192 at T = 2032, k = 16, E = 64
    (dict(T=2032, E=64, n_group=4, topk_group=4, top_k=16), 2),
    (dict(T=2028, E=64, n_group=4, topk_group=4, top_k=16), 4),   # 8177: accepted
    (dict(x=0), 1), (dict(rw=0), 1), (dict(bias=0), 1), (dict(ids=0), 1), (dict(w=0), 1),
    (dict(off=0), 1), (dict(ent=0), 1),
    (dict(x=_A + 4), 1), (dict(rw=_A + 8), 1),      # x, W_r: 16-byte alignment
    (dict(bias=_A + 2), 1), (dict(ids=_A + 2), 1), (dict(w=_A + 1), 1), (dict(off=_A + 2), 1),
    (dict(ent=_A + 3), 1),                          # the rest: 4-byte alignment
])
def test_route_noalloc_refusals(over, code):
    """Each refusal with its documented status; a case just inside a scratch limit passes
    every check and stops at the first CUDA call (no device here: MOE_ERR_CUDA)."""
    a = {**_NOALLOC, **over}
    rc = moe.lib.moe_route_noalloc(a["x"], a["act"], a["T"], a["H"], a["rw"], a["rdt"], a["bias"], a["E"],
                                   a["n_group"], a["topk_group"], a["top_k"], a["rsf"], a["ids"], a["w"],
                                   a["off"], a["ent"], None)
    assert rc == code, (over, rc)


def test_route_noalloc_zero_tokens_is_a_no_op():
    """T = 0 returns MOE_OK with NULL buffers, before any CUDA call."""
    a = {**_NOALLOC, "T": 0}
    rc = moe.lib.moe_route_noalloc(None, a["act"], 0, a["H"], None, a["rdt"], None, a["E"], a["n_group"],
                                   a["topk_group"], a["top_k"], a["rsf"], None, None, None, None, None)
    assert rc == 0


def test_struct_layouts_and_enums_match_the_header(tmp_path):
    """The ctypes structs and constants of the binding against the C compiler's view of
    include/moe_layer.h: size and offset of every field of moe_config and moe_weights, and
    the value of every enum constant the binding mirrors."""
    import json
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    consts = {"MOE_OK": 0, "MOE_ERR_INVALID_ARG": 1, "MOE_ERR_UNSUPPORTED": 2, "MOE_ERR_OOM": 3,
              "MOE_ERR_CUDA": 4, "MOE_ERR_TIMEOUT": 5, "MOE_ERR_DEVICE_CHECK": 6,
              "MOE_W_INT4_G32": moe.W_INT4_G32, "MOE_W_NVFP4": moe.W_NVFP4, "MOE_W_BF16": moe.W_BF16,
              "MOE_W_INT8_ROW": moe.W_INT8_ROW, "MOE_W_INT4_ROW": moe.W_INT4_ROW,
              "MOE_W_INT2_ROW": moe.W_INT2_ROW, "MOE_ACT_NONE": 0, "MOE_ACT_Q8_0": 1,
              "MOE_DT_F32": moe.DT_F32, "MOE_DT_BF16": moe.DT_BF16, "MOE_PATH_AUTO": moe.PATH_AUTO,
              "MOE_PATH_GEMV": moe.PATH_GEMV, "MOE_PATH_GROUPED": moe.PATH_GROUPED,
              "MOE_PATH_GENERIC": moe.PATH_GENERIC}
    assert {v: k for k, v in moe.STATUS.items()} == {k: v for k, v in consts.items() if k.startswith("MOE_OK")
                                                     or k.startswith("MOE_ERR")}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "moe_layer.h"', "int main(void) {",
             'printf("{");']
    for struct, cls in (("moe_config", moe.Config), ("moe_weights", moe.Weights)):
        lines.append(f'printf("\\"{struct}\\": %zu, ", sizeof({struct}));')
        for name, _ in cls._fields_:
            lines.append(f'printf("\\"{struct}.{name}\\": %zu, ", offsetof({struct}, {name}));')
    for name in consts:
        lines.append(f'printf("\\"{name}\\": %d, ", (int){name});')
    lines += ['printf("\\"end\\": 0}\\n");', "return 0; }"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                        "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    c = json.loads(subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout)
    for struct, cls in (("moe_config", moe.Config), ("moe_weights", moe.Weights)):
        assert c[struct] == ctypes.sizeof(cls), struct
        for name, _ in cls._fields_:
            assert c[f"{struct}.{name}"] == getattr(cls, name).offset, (struct, name)
    for name, value in consts.items():
        assert c[name] == value, name


def test_plain_c_consumer(tmp_path):
    """tests/c_abi/host_only.c, a C program that includes the header and links libmoe.so,
    builds with a C compiler and runs its host-only checks (status names, NULL handles,
    argument checks)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    libdir = os.path.dirname(moe.LIB_PATH)
    if not os.path.exists(moe.LIB_PATH):
        pytest.fail("libmoe.so not built")
    exe = tmp_path / "host_only"
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        os.path.join(ROOT, "tests", "c_abi", "host_only.c"), "-L", libdir, "-lmoe",
                        "-Wl,-rpath," + libdir, "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.strip() == "ok", (run.returncode, run.stderr)
