"""GPU parity of the adaptive expert top-p (the pages' "--topp" option; reading in the
oracle's expert_top_p: the shortest score-ordered prefix of the chosen experts reaching p of
their mass, kept weights renormalised to rsf, dropped slots id -1) on every path: the fused
decode kernel (T <= 8), the grouped tcgen05 GEMMs (int4 and NVFP4 on the FP4 tensor cores)
and the generic CUDA-core path; and the GLM-shaped layer at T = 1 over many steps. Routing
(kept sets, weights, grouping) and outputs against the oracle, and the number of dropped
slots is checked to be non-zero so the rule is exercised."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle.moe_oracle import Layer
from synth import LAYERS, make_layer, make_x
from tests.gpu_util import empty_out, out_to_host, x_to_device
from tests.parity import check_out, check_routing

_cache = {}


def get(name, max_tokens=512):
    import quantized_moe_noaux_b300 as moe
    if name not in _cache:
        spec = LAYERS[name]
        arrays = make_layer(spec)
        _cache[name] = (spec, arrays, moe.MoeLayer.from_spec(spec, arrays, max_tokens=max_tokens),
                        Layer.from_spec(spec, arrays))
    return _cache[name]


def check(name, T, step, path, require_drop=True):
    import quantized_moe_noaux_b300 as moe
    spec, arrays, layer, oracle = get(name)
    layer.set_path(path)
    x = make_x(spec, T, step)
    out = empty_out(T, spec.hidden, spec.act_dtype)
    layer.forward(x_to_device(x, spec.act_dtype), out)
    torch.cuda.synchronize()
    assert layer.status() == 0
    got = layer.routing(T)
    layer.set_path(moe.PATH_AUTO)
    ref = oracle.forward(x)
    rep = check_routing(ref, got, bias=arrays["bias"], n_group=spec.n_group,
                        topk_group=spec.topk_group, top_k=spec.top_k, n_experts=spec.n_experts)
    if rep["mismatch"]:
        ref = oracle.forward(x, ids=got["ids"])
    check_out(ref.out, out_to_host(out))
    dropped = int((got["ids"] < 0).sum())
    assert dropped < T * spec.top_k
    if require_drop:
        assert dropped > 0
    return dropped


@pytest.mark.parametrize("T,step", [(3, 1), (8, 2)])
def test_topp_decode_kernel(T, step):
    import quantized_moe_noaux_b300 as moe
    check("small_topp", T, step, moe.PATH_GEMV)


def test_topp_decode_kernel_one_token():
    import quantized_moe_noaux_b300 as moe
    dropped = [check("small_topp", 1, s, moe.PATH_GEMV, require_drop=False) for s in range(8)]
    assert sum(dropped) > 0, dropped


@pytest.mark.parametrize("T,step", [(64, 3), (300, 4)])
def test_topp_grouped_int4(T, step):
    import quantized_moe_noaux_b300 as moe
    check("small_topp", T, step, moe.PATH_GROUPED)


def test_topp_generic():
    import quantized_moe_noaux_b300 as moe
    check("small_topp", 40, 5, moe.PATH_GENERIC)


def test_topp_grouped_nvfp4():
    import quantized_moe_noaux_b300 as moe
    check("small_nvfp4_topp", 300, 6, moe.PATH_GROUPED)


def test_topp_glm_decode_steps():
    """GLM-shaped layer, --topp 0.7, 24 decode steps through the fused kernel: every step's
    routing and output against the oracle; the mean kept experts per token is reported by
    the assertion message if it is not below top_k."""
    import quantized_moe_noaux_b300 as moe
    spec = LAYERS["glm52_topp"]
    arrays = make_layer(spec)
    layer = moe.MoeLayer.from_spec(spec, arrays, max_tokens=1)
    oracle = Layer.from_spec(spec, arrays)
    kept = []
    try:
        for step in range(24):
            x = make_x(spec, 1, step)
            out = empty_out(1, spec.hidden, spec.act_dtype)
            layer.forward(x_to_device(x, spec.act_dtype), out)
            torch.cuda.synchronize()
            assert layer.status() == 0
            got = layer.routing(1)
            ref = oracle.forward(x)
            rep = check_routing(ref, got, bias=arrays["bias"], n_group=spec.n_group,
                                topk_group=spec.topk_group, top_k=spec.top_k, n_experts=spec.n_experts)
            if rep["mismatch"]:
                ref = oracle.forward(x, ids=got["ids"])
            check_out(ref.out, out_to_host(out))
            kept.append(int((got["ids"] >= 0).sum()))
    finally:
        layer.close()
    assert np.mean(kept) < spec.top_k, kept
