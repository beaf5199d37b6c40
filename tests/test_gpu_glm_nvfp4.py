"""GPU parity on the GLM-5.2-shaped NVFP4 layer (H=6144, I=2048, E=256 routed experts as
E2M1 codes with an E4M3 scale per 16 elements and an fp32 tensor scale per matrix; bf16
router and bf16 shared expert; x bf16 quantised per call to NVFP4 for the routed experts):
T=256 with every token's output compared, T=4096 with every token's routing and 320
sampled tokens' outputs. The oracle runs the gate/up projection of the whole batch in both
cases, because the tensor scale of the routed h covers every routed h row of the call."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle.moe_oracle import Layer
from synth import LAYERS, make_layer, make_x
from tests.gpu_util import empty_out, out_to_host, x_to_device
from tests.parity import check_out, check_routing
from tests.test_gpu_nvfp4_act import check_act


@pytest.fixture(scope="module")
def nvfp4_layer():
    import quantized_moe_noaux_b300 as moe
    spec = LAYERS["glm52_nvfp4"]
    arrays = make_layer(spec)
    layer = moe.MoeLayer.from_spec(spec, arrays, max_tokens=4096)
    yield spec, arrays, layer, Layer.from_spec(spec, arrays)
    layer.close()


def run(spec, arrays, layer, oracle, T, step, sample=None):
    x = make_x(spec, T, step)
    out = empty_out(T, spec.hidden, spec.act_dtype)
    layer.forward(x_to_device(x, spec.act_dtype), out)
    torch.cuda.synchronize()
    assert layer.status() == 0
    got = layer.routing(T)
    toks = np.arange(T) if sample is None else np.asarray(sample)
    ref = oracle.forward(x, tokens=toks)
    rep = check_routing(ref, got, bias=arrays["bias"], n_group=spec.n_group,
                        topk_group=spec.topk_group, top_k=spec.top_k, n_experts=spec.n_experts)
    if rep["mismatch"]:
        ref = oracle.forward(x, ids=got["ids"], tokens=toks)
    return check_out(ref.out[toks], out_to_host(out)[toks])


def test_nvfp4_glm_t256_all_tokens(nvfp4_layer):
    spec, arrays, layer, oracle = nvfp4_layer
    run(spec, arrays, layer, oracle, 256, 0)
    # the NVFP4 codes and scales the FP4 tensor cores read, byte for byte
    check_act(spec, layer, make_x(spec, 256, 0), 256)


def test_nvfp4_glm_t4096_sampled(nvfp4_layer):
    spec, arrays, layer, oracle = nvfp4_layer
    rng = np.random.default_rng(4096)
    sample = np.unique(np.concatenate([[0, 4095], rng.choice(4096, 318, replace=False)]))
    run(spec, arrays, layer, oracle, 4096, 1, sample=sample)
