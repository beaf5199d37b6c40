"""GPU parity of the fused decode kernel (T <= 8) on a small layer that still spans many
tiles per CTA (H=2048, I=2048, E=32 + shared, k=4): routing bit-exact and outputs within
tolerance against the oracle, for one token (group-column MMA mode) and 2..8 tokens
(token-column mode); agreement with the generic expert path; repeated calls."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle.moe_oracle import Layer
from synth import LAYERS, make_layer, make_x
from tests.gpu_util import empty_out, out_to_host, x_to_device
from tests.parity import check_out, check_routing


@pytest.fixture(scope="module")
def small():
    import quantized_moe_noaux_b300 as moe
    spec = LAYERS["small"]
    arrays = make_layer(spec)
    layer = moe.MoeLayer.from_spec(spec, arrays, max_tokens=64)
    yield spec, arrays, layer, Layer.from_spec(spec, arrays)
    layer.close()


def run(spec, layer, x, path):
    layer.set_path(path)
    out = empty_out(x.shape[0], spec.hidden, spec.act_dtype)
    n0 = layer.launch_count()
    layer.forward(x_to_device(x, spec.act_dtype), out)
    torch.cuda.synchronize()
    assert layer.status() == 0
    return out, layer.launch_count() - n0


@pytest.mark.parametrize("T,step", [(1, 0), (1, 1), (2, 2), (3, 3), (5, 4), (8, 5)])
def test_decode_parity(small, T, step):
    import quantized_moe_noaux_b300 as moe
    spec, arrays, layer, oracle = small
    x = make_x(spec, T, step)
    out, launches = run(spec, layer, x, moe.PATH_GEMV)
    assert launches == 1                       # one fused kernel
    got = layer.routing(T)
    ref = oracle.forward(x)
    rep = check_routing(ref, got, bias=arrays["bias"], n_group=spec.n_group,
                        topk_group=spec.topk_group, top_k=spec.top_k, n_experts=spec.n_experts)
    if rep["mismatch"]:
        ref = oracle.forward(x, ids=got["ids"])
    check_out(ref.out, out_to_host(out))
    layer.set_path(moe.PATH_AUTO)


def test_decode_matches_generic_path_and_repeats(small):
    import quantized_moe_noaux_b300 as moe
    spec, _, layer, _ = small
    for T, step in [(1, 7), (4, 8)]:
        x = make_x(spec, T, step)
        a, _ = run(spec, layer, x, moe.PATH_GEMV)
        b, _ = run(spec, layer, x, moe.PATH_GROUPED)
        c, _ = run(spec, layer, x, moe.PATH_GEMV)   # the counters were reset by the last call
        ha, hb, hc = out_to_host(a), out_to_host(b), out_to_host(c)
        rel = np.linalg.norm(ha - hb) / np.linalg.norm(hb)
        assert rel < 2e-3, rel
        assert np.allclose(ha, hc, rtol=0, atol=2e-3 * np.abs(ha).max())
    layer.set_path(moe.PATH_AUTO)


def test_decode_path_refuses_large_t(small):
    import quantized_moe_noaux_b300 as moe
    spec, _, layer, _ = small
    layer.set_path(moe.PATH_GEMV)
    x = make_x(spec, 9, 0)
    with pytest.raises(moe.MoeError):
        layer.forward(x_to_device(x, spec.act_dtype), empty_out(9, spec.hidden, spec.act_dtype))
    layer.set_path(moe.PATH_AUTO)


def test_decode_wait_timeout_and_recovery(small):
    """With a wait limit of 0 the fused kernel's waits on other CTAs give up at once: the
    forward ends (no hang) and the status word reports MOE_ERR_TIMEOUT. With the limit
    restored and the status cleared, the next two forwards are correct again (the aborted
    call left no stale counters behind)."""
    import quantized_moe_noaux_b300 as moe
    spec, arrays, layer, oracle = small
    layer.set_path(moe.PATH_GEMV)
    x = make_x(spec, 1, 21)
    out = empty_out(1, spec.hidden, spec.act_dtype)
    layer.set_wait_limit(0)
    layer.forward(x_to_device(x, spec.act_dtype), out)
    torch.cuda.synchronize()
    assert layer.status() == 5            # MOE_ERR_TIMEOUT
    layer.set_wait_limit(2_000_000_000)
    layer.reset_status()
    for T, step in [(1, 22), (3, 23)]:
        x = make_x(spec, T, step)
        out, _ = run(spec, layer, x, moe.PATH_GEMV)
        got = layer.routing(T)
        ref = oracle.forward(x)
        rep = check_routing(ref, got, bias=arrays["bias"], n_group=spec.n_group,
                            topk_group=spec.topk_group, top_k=spec.top_k, n_experts=spec.n_experts)
        if rep["mismatch"]:
            ref = oracle.forward(x, ids=got["ids"])
        check_out(ref.out, out_to_host(out))
    layer.set_path(moe.PATH_AUTO)
