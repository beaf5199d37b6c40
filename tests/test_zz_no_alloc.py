"""moe_route_noalloc: routing for callers that cannot allocate device memory.

The entry point keeps its kernels' scratch in a fixed file-scope device array instead of
memory from cudaMalloc. Its results must equal the routing the layer entry point
(moe_layer_forward + moe_layer_get_routing) computes for the same inputs, on two calls
in a row (the second call reuses the array the first one left behind). This file is
collected last so a failure here stops a -x run only after every other test ran.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from synth import LAYERS, make_layer, make_x
from tests.gpu_util import empty_out, x_to_device

_DT = {"f32": 0, "bf16": 1}


def _noalloc(lib, spec, xd, wr, bias, T, stream):
    k, E = spec.top_k, spec.n_experts
    ids = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), -1.0, dtype=torch.float32, device="cuda")
    off = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    ent = torch.full((T * k,), -1, dtype=torch.int32, device="cuda")
    rc = lib.moe_route_noalloc(xd.data_ptr(), _DT[spec.act_dtype], T, spec.hidden, wr.data_ptr(),
                               _DT[spec.router_dtype], bias.data_ptr(), E, spec.n_group,
                               spec.topk_group, k, spec.rsf, ids.data_ptr(), w.data_ptr(),
                               off.data_ptr(), ent.data_ptr(), stream)
    return rc, ids, w, off, ent


def test_noalloc_routing_matches_layer_entry_point():
    import quantized_moe_noaux_b300 as moe
    lib = moe.lib
    spec = LAYERS["tiny"]
    arrays = make_layer(spec)
    layer = moe.MoeLayer.from_spec(spec, arrays, max_tokens=8175)
    wr = torch.from_numpy(np.array(arrays["router_w"])).cuda()
    bias = torch.from_numpy(np.array(arrays["bias"])).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    # two calls in a row with the row router, one with the tiled router (T >= 128), and the
    # largest T whose grouping work list fits the scratch (T + E + 1 = 8192 items at k = 4)
    for T, step in [(37, 11), (64, 12), (256, 13), (8175, 14)]:
        x = make_x(spec, T, step)
        xd = x_to_device(x, spec.act_dtype)
        out = empty_out(T, spec.hidden, spec.act_dtype)
        layer.forward(xd, out)
        ref = layer.routing(T)
        rc, ids, w, off, ent = _noalloc(lib, spec, xd, wr, bias, T, stream)
        assert rc == 0, moe.STATUS.get(rc, rc)
        torch.cuda.synchronize()
        assert np.array_equal(ids.cpu().numpy(), ref["ids"])
        assert np.allclose(w.cpu().numpy(), ref["weights"], rtol=1e-5, atol=0)
        assert np.array_equal(off.cpu().numpy(), ref["offsets"])
        assert np.array_equal(ent.cpu().numpy(), ref["entries"])
    layer.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import quantized_moe_noaux_b300 as moe
    spec = LAYERS["glm52"]
    # T * E = 2048 * 256 > 262144 logits: refused before any work is enqueued
    rc = moe.lib.moe_route_noalloc(1 << 20, 1, 2048, spec.hidden, 1 << 20, 0, 1 << 20,
                                   spec.n_experts, spec.n_group, spec.topk_group, spec.top_k,
                                   spec.rsf, 1 << 20, 1 << 20, 1 << 20, 1 << 20, None)
    assert rc == 2   # MOE_ERR_UNSUPPORTED


def test_noalloc_bf16_activations_match_within_near_ties():
    """bf16 activations with an fp32 router: the layer computes the logits on the tensor
    cores, this entry point on the CUDA cores, so their sums are rounded differently. Every
    token whose selection margin (fp64) exceeds the near-tie bound gets the same experts
    and weights within 1e-5; the grouping is the same wherever the selections agree."""
    import quantized_moe_noaux_b300 as moe
    from oracle.moe_oracle import Layer
    from tests.parity import NEAR_TIE
    lib = moe.lib
    spec = LAYERS["small"]
    arrays = make_layer(spec)
    layer = moe.MoeLayer.from_spec(spec, arrays, max_tokens=256)
    oracle = Layer.from_spec(spec, arrays)
    wr = torch.from_numpy(np.array(arrays["router_w"])).cuda()
    bias = torch.from_numpy(np.array(arrays["bias"])).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    for T, step in [(64, 21), (256, 22)]:
        x = make_x(spec, T, step)
        xd = x_to_device(x, spec.act_dtype)
        out = empty_out(T, spec.hidden, spec.act_dtype)
        layer.forward(xd, out)
        ref = layer.routing(T)
        rc, ids, w, off, ent = _noalloc(lib, spec, xd, wr, bias, T, stream)
        assert rc == 0, moe.STATUS.get(rc, rc)
        torch.cuda.synchronize()
        ids, w = ids.cpu().numpy(), w.cpu().numpy()
        _, sel = oracle.route(oracle.widen_x(x))
        same = np.array([sorted(ids[t]) == sorted(ref["ids"][t]) for t in range(T)])
        assert np.all(same | (sel.margin <= NEAR_TIE))
        for t in np.nonzero(same)[0]:
            ra = dict(zip(ref["ids"][t].tolist(), ref["weights"][t].tolist()))
            for e, wv in zip(ids[t].tolist(), w[t].tolist()):
                assert abs(wv - ra[e]) <= 1e-5 * abs(ra[e])
        if same.all():
            assert np.array_equal(off.cpu().numpy(), ref["offsets"])
            assert np.array_equal(ent.cpu().numpy(), ref["entries"])
    layer.close()


def test_noalloc_rejects_misaligned_activations():
    """x must be 16-byte aligned (the tiled router reads it 16 bytes at a time): an offset
    view is refused before anything is enqueued."""
    import quantized_moe_noaux_b300 as moe
    spec = LAYERS["tiny"]
    arrays = make_layer(spec)
    wr = torch.from_numpy(np.array(arrays["router_w"])).cuda()
    bias = torch.from_numpy(np.array(arrays["bias"])).cuda()
    x = torch.zeros((257, spec.hidden), dtype=torch.float32, device="cuda").view(-1)[1:1 + 256 * spec.hidden]
    stream = torch.cuda.current_stream().cuda_stream
    k, E, T = spec.top_k, spec.n_experts, 256
    outs = [torch.empty(n, dtype=dt, device="cuda") for n, dt in
            ((T * k, torch.int32), (T * k, torch.float32), (E + 1, torch.int32), (T * k, torch.int32))]
    rc = moe.lib.moe_route_noalloc(x.data_ptr(), 0, T, spec.hidden, wr.data_ptr(), 0, bias.data_ptr(), E,
                                   spec.n_group, spec.topk_group, k, spec.rsf, *[o.data_ptr() for o in outs],
                                   stream)
    assert rc == 1   # MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
