"""The seeded input generator: container encoders checked against the oracle's
decoders and the formats' error bounds; draws are reproducible and pool-independent."""

import numpy as np
import torch

from oracle import moe_oracle as O
from synth import (LAYERS, WORKLOADS, bf16_bits_to_f32, f32_to_bf16_bits, make_layer, make_x,
                   quantize_int4_g32, quantize_nvfp4_weight)
from synth.layer import _draw_expert


def test_bf16_rounding_matches_torch():
    v = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 100
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(f32_to_bf16_bits(v), ref)
    assert np.array_equal(bf16_bits_to_f32(ref), torch.from_numpy(ref.view(np.int16))
                          .view(torch.bfloat16).float().numpy())


def test_int4_g32_half_step_bound():
    rng = np.random.default_rng(1)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    w[3, 32:64] = 0.0                          # an all-zero group
    codes, scales = quantize_int4_g32(w)
    deq = O.dequant_int4_g32(codes, scales)
    s = np.repeat(scales.astype(np.float64), 32, axis=1)
    assert np.all(np.abs(deq - w) <= s / 2 + 1e-30)
    assert np.all(deq[3, 32:64] == 0) and np.all(scales[3, 1] == 0)
    c = O.decode_int4(codes).reshape(64, 8, 32)
    nz = scales.astype(np.float64) != 0
    assert np.all(np.abs(c).max(axis=2)[nz] == 7)     # the group absmax maps to +-7
    assert np.array_equal(scales, (np.abs(w.reshape(64, 8, 32)).max(2) / np.float32(7))
                          .astype(np.float16))


def test_nvfp4_weight_bound_and_roundtrip():
    rng = np.random.default_rng(2)
    w = (rng.standard_normal((32, 128)) * 0.02).astype(np.float32)
    codes, scales, ts = quantize_nvfp4_weight(w)
    deq = O.dequant_nvfp4(codes, scales, ts)
    unit = np.repeat(O.decode_e4m3(scales), 16, axis=1) * float(ts)
    mag = np.abs(deq) / np.where(unit == 0, 1, unit)
    # half the E2M1 spacing at the chosen code: 0.25 below 2, 0.5 below 4, 1 above;
    # saturation at 6 may add the block scale's own rounding (<= 2^-4 relative)
    half = np.where(mag < 2, 0.25, np.where(mag < 4, 0.5, 1.0)) * unit
    assert np.all(np.abs(deq - w) <= half * (1 + 2 ** -3) + 1e-30)
    # values already on the grid come back (to the fp32 rounding of amax / 2688)
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -6, -4, -3, -2, -1.5, -1, -.5, 0], np.float32)
    g = np.tile(grid, (4, 2)) * np.float32(1.0)
    codes, scales, ts = quantize_nvfp4_weight(g)
    assert np.allclose(O.dequant_nvfp4(codes, scales, ts), g, rtol=1e-7, atol=0)
    assert np.array_equal(O.decode_e2m1(np.stack([codes & 15, codes >> 4], -1).reshape(4, 32)), g)


def test_layer_shapes_and_reproducible():
    spec = LAYERS["tiny"]
    a = make_layer(spec)
    E, H, I = spec.n_experts, spec.hidden, spec.inter
    assert a["router_w"].shape == (E, H) and a["bias"].shape == (E,)
    assert a["gu_codes"].shape == (E, 2 * I, H // 2) and a["gu_scales"].shape == (E, 2 * I, H // 32)
    assert a["d_codes"].shape == (E, H, I // 2) and a["d_scales"].shape == (E, H, I // 32)
    assert a["sh_gu_codes"].shape == (1, 2 * I, H // 2)
    # pool draw equals serial draw
    b = make_layer.__wrapped__(spec, workers=2)
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    # expert e of the layer is stream [seed, 2, e]
    res = _draw_expert((spec.seed, 5, H, I, spec.weight_std, "int4_g32"))
    assert np.array_equal(res["gu_codes"], a["gu_codes"][5])
    x1, x2 = make_x(spec, 4, 0), make_x(spec, 4, 0)
    assert np.array_equal(x1, x2) and not np.array_equal(x1, make_x(spec, 4, 1))


def test_workload_table():
    assert WORKLOADS["glm52_decode_t1"].tokens == 1
    assert WORKLOADS["glm52_prefill_t2048"].layer.bias_std == 0.5
    assert WORKLOADS["glm52_decode_t32"].layer.bias_std == 0.0
    nv = WORKLOADS["glm52_nvfp4_t4096"].layer
    assert (nv.weight_format, nv.router_dtype, nv.shared_format) == ("nvfp4", "bf16", "bf16")


def test_bias_swap_equals_fresh_draw():
    from dataclasses import replace
    from synth import with_bias_of
    base = LAYERS["tiny"]
    other = replace(base, name="tiny_bias0.5", bias_std=0.5)
    a = with_bias_of(make_layer(base), other)
    b = make_layer(other)
    for k in b:
        assert np.array_equal(a[k], b[k]), k
