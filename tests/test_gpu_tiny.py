"""GPU parity on the tiny layer (H=256, I=128, E=16, k=4, fp32 activations): routing
bit-exact, outputs within tolerance, across token counts with ragged tails."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle.moe_oracle import Layer
from synth import LAYERS, make_layer, make_x
from tests.gpu_util import empty_out, out_to_host, x_to_device
from tests.parity import check_out, check_routing


@pytest.fixture(scope="module")
def tiny():
    import quantized_moe_noaux_b300 as moe
    spec = LAYERS["tiny"]
    arrays = make_layer(spec)
    layer = moe.MoeLayer.from_spec(spec, arrays, max_tokens=512)
    yield spec, arrays, layer, Layer.from_spec(spec, arrays)
    layer.close()


def run_and_check(spec, layer, oracle, T, step):
    x = make_x(spec, T, step)
    xd = x_to_device(x, spec.act_dtype)
    out = empty_out(T, spec.hidden, spec.act_dtype)
    layer.forward(xd, out)
    torch.cuda.synchronize()
    assert layer.status() == 0
    got = layer.routing(T)
    ref = oracle.forward(x)
    rep = check_routing(ref, got, bias=oracle.a["bias"], n_group=spec.n_group,
                        topk_group=spec.topk_group, top_k=spec.top_k, n_experts=spec.n_experts)
    if rep["mismatch"]:
        ref = oracle.forward(x, ids=got["ids"])
    return check_out(ref.out, out_to_host(out))


@pytest.mark.parametrize("T,step", [(1, 0), (4, 0), (5, 1), (37, 2), (64, 3), (255, 4), (512, 5)])
def test_tiny_parity(tiny, T, step):
    spec, _, layer, oracle = tiny
    run_and_check(spec, layer, oracle, T, step)


def test_tiny_forward_host_matches_device(tiny):
    spec, _, layer, _ = tiny
    x = make_x(spec, 13, 7)
    xd = x_to_device(x, spec.act_dtype)
    out = empty_out(13, spec.hidden, spec.act_dtype)
    layer.forward(xd, out)
    torch.cuda.synchronize()
    host_out = np.empty((13, spec.hidden), np.float32)
    layer.forward_host(np.ascontiguousarray(x), host_out)
    # the generic path combines with fp32 atomics, so summation order may differ by run
    dev = out.cpu().numpy()
    assert np.allclose(dev, host_out, rtol=1e-5, atol=1e-6 * np.abs(dev).max())


def test_tiny_zero_tokens_and_bad_args(tiny):
    import quantized_moe_noaux_b300 as moe
    spec, _, layer, _ = tiny
    x = torch.zeros((0, spec.hidden), device="cuda")
    out = torch.zeros((0, spec.hidden), device="cuda")
    layer.forward(x, out)                       # T = 0 is a no-op
    big = torch.zeros((513, spec.hidden), device="cuda")
    with pytest.raises(moe.MoeError):
        layer.forward(big, big.clone())        # T > max_tokens
    assert moe.lib.moe_layer_forward(layer.handle, None, 4, None, None) == 1
    torch.cuda.synchronize()
    assert layer.status() == 0
