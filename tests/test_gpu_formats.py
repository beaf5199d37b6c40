"""GPU parity of the pages' per-row weight formats (int8, packed int4, packed int2 with one
fp32 scale per row) and of Q8_0-style int8 activations, on the CUDA-core batch-union
kernels (the path these formats run on): small layers (H = I = 2048, E = 32 + 1 shared,
k = 4), one token, a ragged batch and a batch of many chunks; routing and outputs against
the oracle."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle.moe_oracle import Layer
from synth import LAYERS, make_layer, make_x
from tests.gpu_util import empty_out, out_to_host, x_to_device
from tests.parity import check_out, check_routing

_cache = {}


def get(name):
    import quantized_moe_noaux_b300 as moe
    if name not in _cache:
        spec = LAYERS[name]
        arrays = make_layer(spec)
        _cache[name] = (spec, arrays, moe.MoeLayer.from_spec(spec, arrays, max_tokens=128),
                        Layer.from_spec(spec, arrays))
    return _cache[name]


@pytest.mark.parametrize("name", ["small_int8_row", "small_int4_row", "small_int2_row", "small_int4_row_q8"])
@pytest.mark.parametrize("T,step", [(1, 0), (9, 1), (67, 2)])
def test_row_formats(name, T, step):
    spec, arrays, layer, oracle = get(name)
    x = make_x(spec, T, step)
    out = empty_out(T, spec.hidden, spec.act_dtype)
    layer.forward(x_to_device(x, spec.act_dtype), out)
    torch.cuda.synchronize()
    assert layer.status() == 0
    got = layer.routing(T)
    ref = oracle.forward(x)
    rep = check_routing(ref, got, bias=arrays["bias"], n_group=spec.n_group,
                        topk_group=spec.topk_group, top_k=spec.top_k, n_experts=spec.n_experts)
    if rep["mismatch"]:
        ref = oracle.forward(x, ids=got["ids"])
    check_out(ref.out, out_to_host(out))


def test_row_format_paths_rejected():
    """GEMV and GROUPED do not take the per-row formats: MOE_ERR_UNSUPPORTED."""
    import quantized_moe_noaux_b300 as moe
    spec, _, layer, _ = get("small_int4_row")
    x = x_to_device(make_x(spec, 2, 0), spec.act_dtype)
    out = empty_out(2, spec.hidden, spec.act_dtype)
    for path in (moe.PATH_GEMV, moe.PATH_GROUPED):
        layer.set_path(path)
        with pytest.raises(moe.MoeError) as ei:
            layer.forward(x, out)
        assert ei.value.code == 2
    layer.set_path(moe.PATH_AUTO)
