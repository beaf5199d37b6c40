"""Exact-arithmetic GPU cases: every path's output equals the oracle's bit for bit.

With the test-only identity activation (h = gate * up, on the GPU through
moe_layer_set_test_activation and in the oracle through Layer.forward(activation=
"identity")), inputs can be chosen so that no operation of either side rounds:
- router weights 0: every logit is 0 and every gate score sigmoid(0) = 1/2, the dyadic
  biases -e/1024 select experts 0-3 (groups 0 and 1), and each weight is exactly
  rsf / k = 0.625;
- int4 codes in {-1, 0, 1} with group scales 1/4 (exact in fp16), x fp32 with 8 entries
  of +-1 per token: gate and up are multiples of 1/4 below 2 in magnitude, h multiples of
  1/16 below 4 (exact in fp16), y multiples of 1/64 below 2^11, the combine multiples of
  1/512 below 2^13: all exact in fp32, in any summation order, and in fp16 where the fast
  paths store operands.
So the fused decode kernel (one token on CUDA cores, four tokens on the tensor cores), the
grouped tcgen05 path and the generic path must all reproduce the oracle exactly."""

from dataclasses import replace

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle.moe_oracle import Layer
from synth import LAYERS
from tests.gpu_util import empty_out, out_to_host, x_to_device

SPEC = replace(LAYERS["small"], name="small_exact", act_dtype="f32", router_dtype="f32")


def pack_nibbles(codes):
    u = (codes.astype(np.int8).view(np.uint8) & 0x0F).reshape(codes.shape[:-1] + (-1, 2))
    return (u[..., 0] | (u[..., 1] << 4)).astype(np.uint8)


def exact_arrays(seed=0):
    rng = np.random.default_rng(seed)
    H, I, E = SPEC.hidden, SPEC.inter, SPEC.n_experts

    def expert(n):
        gu = rng.integers(-1, 2, (n, 2 * I, H))
        d = rng.integers(-1, 2, (n, H, I))
        return {"gu_codes": pack_nibbles(gu), "gu_scales": np.full((n, 2 * I, H // 32), 0.25, np.float16),
                "d_codes": pack_nibbles(d), "d_scales": np.full((n, H, I // 32), 0.25, np.float16)}

    a = {"router_w": np.zeros((E, H), np.float32),
         "bias": (-np.arange(E, dtype=np.float32) / np.float32(1024.0))}
    a.update(expert(E))
    a.update({"sh_" + k: v for k, v in expert(1).items()})
    return a


def exact_x(T, seed):
    rng = np.random.default_rng(1000 + seed)
    x = np.zeros((T, SPEC.hidden), np.float32)
    for t in range(T):
        pos = rng.choice(SPEC.hidden, 8, replace=False)
        x[t, pos] = rng.choice([-1.0, 1.0], 8)
    return x


_cache = {}


def layer_and_oracle():
    import quantized_moe_noaux_b300 as moe
    if "l" not in _cache:
        arrays = exact_arrays()
        layer = moe.MoeLayer.from_spec(SPEC, arrays, max_tokens=64)
        layer.set_test_activation(True)
        _cache["l"] = (arrays, layer, Layer.from_spec(SPEC, arrays))
    return _cache["l"]


@pytest.mark.parametrize("path_name,T", [("gemv", 1), ("gemv", 4), ("grouped", 24), ("generic", 5)])
def test_identity_activation_bit_exact(path_name, T):
    import quantized_moe_noaux_b300 as moe
    path = {"gemv": moe.PATH_GEMV, "grouped": moe.PATH_GROUPED, "generic": moe.PATH_GENERIC}[path_name]
    arrays, layer, oracle = layer_and_oracle()
    x = exact_x(T, T)
    layer.set_path(path)
    out = empty_out(T, SPEC.hidden, SPEC.act_dtype)
    layer.forward(x_to_device(x, SPEC.act_dtype), out)
    torch.cuda.synchronize()
    assert layer.status() == 0
    layer.set_path(moe.PATH_AUTO)
    got = out_to_host(out)
    ref = oracle.forward(x, activation="identity")
    assert sorted(layer.routing(T)["ids"][0].tolist()) == [0, 1, 2, 3]
    assert np.all(layer.routing(T)["weights"] == np.float32(0.625))
    assert np.abs(ref.out).max() > 1.0          # a non-trivial output
    bad = np.argwhere(got != ref.out)
    assert bad.size == 0, (len(bad), bad[:4].tolist(), got[tuple(bad[0])], ref.out[tuple(bad[0])])


def test_silu_restored():
    """Switching the identity off gives the SiLU layer again (within the usual tolerance)."""
    import quantized_moe_noaux_b300 as moe
    from tests.parity import check_out
    arrays, layer, oracle = layer_and_oracle()
    x = exact_x(3, 9)
    layer.set_test_activation(False)
    try:
        out = empty_out(3, SPEC.hidden, SPEC.act_dtype)
        layer.forward(x_to_device(x, SPEC.act_dtype), out)
        torch.cuda.synchronize()
        check_out(oracle.forward(x).out, out_to_host(out))
    finally:
        layer.set_test_activation(True)
