"""GPU parity on exact router ties. With W_r = 0 every logit is exactly 0 and every sigmoid
score exactly 1/2 on both sides, and dyadic biases keep the biased scores exact in fp32 and
fp64. The bias draw below ties three groups at the kept-group boundary and five experts at
the top-k boundary (both oracle margins are exactly 0). So the lower-index rule for groups
and for experts decides the selection, and every path must return the oracle's ids bit for
bit, with weights of exactly rsf / top_k: the fused decode kernel (warp selection), the
grouped path (tensor-core router) and the generic path."""

import numpy as np
import pytest
import torch

from oracle.moe_oracle import Layer, select_experts
from synth import LAYERS, make_layer, make_x
from tests.gpu_util import empty_out, out_to_host, x_to_device
from tests.parity import check_out

_BIAS_VALUES = np.array([-0.25, 0.0, 0.125, 0.25], dtype=np.float32)


def _tied_bias(n_experts):
    return np.random.default_rng(0).choice(_BIAS_VALUES, size=n_experts).astype(np.float32)


def test_tie_fixture_is_tied():
    """The oracle's selection for these scores (all 1/2) ties at both boundaries."""
    spec = LAYERS["small"]
    sel = select_experts(np.full((1, spec.n_experts), 0.5), _tied_bias(spec.n_experts), spec.n_group,
                         spec.topk_group, spec.top_k)
    assert sel.group_margin[0] == 0.0 and sel.expert_margin[0] == 0.0
    assert sorted(sel.ids[0].tolist()) == [9, 11, 14, 19]   # groups 1, 2 of the tied 1, 2, 3


@pytest.fixture(scope="module")
def tied():
    import quantized_moe_noaux_b300 as moe
    spec = LAYERS["small"]
    arrays = dict(make_layer(spec))
    arrays["router_w"] = np.zeros_like(arrays["router_w"])
    arrays["bias"] = _tied_bias(spec.n_experts)
    layer = moe.MoeLayer.from_spec(spec, arrays, max_tokens=64)
    yield spec, arrays, layer, Layer.from_spec(spec, arrays)
    layer.close()


@pytest.mark.gpu
@pytest.mark.parametrize("path,T", [("GEMV", 1), ("GEMV", 4), ("GROUPED", 16), ("GENERIC", 16)])
def test_exact_ties_take_lower_index(tied, path, T):
    import quantized_moe_noaux_b300 as moe
    spec, _, layer, oracle = tied
    layer.set_path(getattr(moe, "PATH_" + path))
    x = make_x(spec, T, 40 + T)
    out = empty_out(T, spec.hidden, spec.act_dtype)
    layer.forward(x_to_device(x, spec.act_dtype), out)
    torch.cuda.synchronize()
    assert layer.status() == 0
    got = layer.routing(T)
    ref = oracle.forward(x)
    for t in range(T):
        assert sorted(got["ids"][t].tolist()) == sorted(ref.ids[t].tolist()), (path, t)
    np.testing.assert_array_equal(got["weights"], np.full((T, spec.top_k), spec.rsf / spec.top_k, np.float32))
    check_out(ref.out, out_to_host(out))
    layer.set_path(moe.PATH_AUTO)
