"""moe_cache_slots_for_memory on the CPU (host arithmetic only): the expert slots of a
cached layer that fit a memory budget, the shared expert's slot included. One int4-g32
expert of the GLM-shaped layer packs to 21,233,664 bytes (2I x H gate/up plus H x I down
codes at half a byte and an fp16 scale per 32), the same as its row-major store."""

import ctypes
from dataclasses import replace

import pytest

import quantized_moe_noaux_b300 as moe
from synth import LAYERS

B_E = 21_233_664
GLM = LAYERS["glm52"]


def test_glm_expert_size_and_budgets():
    assert moe.cache_slots_for_memory(GLM, 1, 33 * B_E) == 32          # 32 routed + shared
    assert moe.cache_slots_for_memory(GLM, 1, 33 * B_E - 1) == 31
    assert moe.cache_slots_for_memory(GLM, 1, 10 * B_E) == 9            # the minimum is 8 (T*k)
    assert moe.cache_slots_for_memory(GLM, 1, 1 << 62) == GLM.n_experts  # capped at E


def test_budget_below_the_minimum_is_oom():
    with pytest.raises(moe.MoeError) as ei:
        moe.cache_slots_for_memory(GLM, 1, 9 * B_E - 1)                 # 8 routed + shared needed
    assert ei.value.code == 3
    with pytest.raises(moe.MoeError) as ei:
        moe.cache_slots_for_memory(GLM, 64, 257 * B_E - 1)              # 64 tokens need all 256
    assert ei.value.code == 3
    assert moe.cache_slots_for_memory(GLM, 64, 257 * B_E) == 256


def test_configurations_a_cached_layer_does_not_take():
    for spec in (LAYERS["glm52_nvfp4"] if "glm52_nvfp4" in LAYERS else replace(GLM, weight_format="nvfp4"),
                 replace(GLM, act_quant="q8_0"), replace(GLM, weight_format="int4_row", shared_format="int4_row")):
        with pytest.raises(moe.MoeError) as ei:
            moe.cache_slots_for_memory(spec, 1, 1 << 40)
        assert ei.value.code == 2, spec.name
    with pytest.raises(moe.MoeError) as ei:
        moe.cache_slots_for_memory(replace(GLM, hidden=0), 1, 1 << 40)
    assert ei.value.code == 1


def test_null_pointers_and_zeroed_result():
    slots = ctypes.c_int32(77)
    assert moe.lib.moe_cache_slots_for_memory(None, 1 << 40, ctypes.byref(slots)) == 1
    assert slots.value == 0
    cfg = moe.config_from_spec(GLM, 1)
    assert moe.lib.moe_cache_slots_for_memory(ctypes.byref(cfg), 1 << 40, None) == 1
    slots = ctypes.c_int32(77)
    assert moe.lib.moe_cache_slots_for_memory(ctypes.byref(cfg), 0, ctypes.byref(slots)) == 3
    assert slots.value == 0
