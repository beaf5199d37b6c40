"""Failure detection without a GPU fault: the device routing checks (a sanitizer substitute,
reporting MOE_ERR_DEVICE_CHECK through the status word instead of trapping) and forced
allocation failures at creation (MOE_ERR_OOM, everything released).

The checks run on valid routings of every path (status stays clean) and on routings with
planted mistakes, which the checker reads only within the arrays' bounds."""


import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from synth import LAYERS, make_layer, make_x
from tests.gpu_util import empty_out, x_to_device


def run(layer, spec, T, step, path):
    import quantized_moe_noaux_b300 as moe
    layer.set_path(path)
    out = empty_out(T, spec.hidden, spec.act_dtype)
    layer.forward(x_to_device(make_x(spec, T, step), spec.act_dtype), out)
    torch.cuda.synchronize()
    layer.set_path(moe.PATH_AUTO)
    return layer.status()


@pytest.mark.parametrize("name,T,path_name", [("small", 1, "gemv"), ("small", 6, "gemv"), ("small", 80, "grouped"),
                                              ("small", 20, "generic"), ("small_topp", 40, "grouped"),
                                              ("small_nvfp4", 50, "grouped")])
def test_debug_checks_pass_on_valid_routing(name, T, path_name):
    import quantized_moe_noaux_b300 as moe
    spec = LAYERS[name]
    layer = moe.MoeLayer.from_spec(spec, make_layer(spec), max_tokens=128)
    try:
        layer.set_debug_checks(True)
        path = {"gemv": moe.PATH_GEMV, "grouped": moe.PATH_GROUPED, "generic": moe.PATH_GENERIC}[path_name]
        assert run(layer, spec, T, 3, path) == 0
    finally:
        layer.close()


def _check(ids, offsets, entries, T, k, E):
    import quantized_moe_noaux_b300 as moe
    d = [torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda() for a in (ids, offsets, entries)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = moe.lib.moe_check_routing(d[0].data_ptr(), d[1].data_ptr(), d[2].data_ptr(), T, k, E,
                                   status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    return int(status.item())


def test_check_routing_catches_planted_mistakes():
    import quantized_moe_noaux_b300 as moe
    spec = LAYERS["small"]
    layer = moe.MoeLayer.from_spec(spec, make_layer(spec), max_tokens=64)
    try:
        T, k, E = 40, spec.top_k, spec.n_experts
        assert run(layer, spec, T, 5, moe.PATH_GROUPED) == 0
        r = layer.routing(T)
        ids, off, ent = r["ids"].ravel(), r["offsets"], r["entries"]
        assert _check(ids, off, ent, T, k, E) == 0
        e0 = int(np.flatnonzero(np.diff(off) >= 2)[0])     # an expert with two or more entries
        mutants = {}
        m = ids.copy(); m[3] = E; mutants["id out of range"] = (m, off, ent)
        m = off.copy(); m[e0 + 1] = m[e0] - 1; mutants["offsets decrease"] = (ids, m, ent)
        m = off.copy(); m[E] -= 1; mutants["offsets end short"] = (ids, m, ent)
        m = off.copy(); m[E] = T * k + 1000; mutants["offsets end past the slots"] = (ids, m, ent)
        m = ent.copy(); m[off[e0]], m[off[e0] + 1] = m[off[e0] + 1], m[off[e0]]; mutants["tokens out of order"] = (ids, off, m)
        m = ent.copy(); m[off[e0]] = (m[off[e0]] // k) * k + (m[off[e0]] + 1) % k; mutants["entry of another slot"] = (ids, off, m)
        m = ent.copy(); m[0] = -7; mutants["entry out of range"] = (ids, off, m)
        for what, (a, b, c) in mutants.items():
            assert _check(a, b, c, T, k, E) == 6, what     # MOE_ERR_DEVICE_CHECK
    finally:
        layer.close()


def test_forced_allocation_failure_releases_everything():
    import quantized_moe_noaux_b300 as moe
    spec = LAYERS["small"]
    arrays = make_layer(spec)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    try:
        for nth in (1, 2, 3, 7, 15, 25):
            assert moe.lib.moe_test_fail_allocation(nth) == 0
            with pytest.raises(moe.MoeError) as ei:
                moe.MoeLayer.from_spec(spec, arrays, max_tokens=64)
            assert ei.value.code == 3, nth                   # MOE_ERR_OOM
            torch.cuda.synchronize()
            assert abs(torch.cuda.mem_get_info()[0] - free0) < 64 << 20, nth   # nothing held
    finally:
        moe.lib.moe_test_fail_allocation(0)
    layer = moe.MoeLayer.from_spec(spec, arrays, max_tokens=64)
    assert run(layer, spec, 4, 1, moe.PATH_AUTO) == 0
    layer.close()
