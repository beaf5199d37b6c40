"""Byte-exact NVFP4 activation quantiser on the GPU ("NVIDIA stellt neues GLM-5.2 NVFP4 Modell
vor", section "Technische Details und Quantisierungsansatz": E2M1 elements, one E4M3 scale per
16 elements, an fp32 tensor scale). The layer quantises x once per call for its block-scaled
FP4 GEMM; the codes and scales it fed the tensor cores (expert-sorted routed rows) are read
back and compared byte for byte with the oracle's quantiser on the same x. Every E2M1 code
and E4M3 scale is decided by fp32 divisions on both sides, so they must agree exactly; the
one freedom is the sign bit of a zero code. Also the degenerate all-zero x (tensor scale 0:
zero scales and codes, output = the shared expert of zero = 0)."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle.moe_oracle import Layer, decode_e2m1, decode_e4m3, nvfp4_activation_parts
from synth import LAYERS, make_layer, make_x
from tests.gpu_util import empty_out, out_to_host, x_to_device
from tests.parity import check_out

_E2M1 = decode_e2m1(np.arange(16))            # value of each nibble
_E4M3 = decode_e4m3(np.arange(0x7F))          # value of each non-negative finite byte


def expected_bytes(code_val: np.ndarray, sb: np.ndarray):
    """Oracle values -> storage: nibble of each signed E2M1 value (positive zero), byte of
    each E4M3 scale (table lookup; both tables are bijective on these values)."""
    mag = np.abs(code_val)
    idx = np.searchsorted(_E2M1[:8], mag)
    assert np.array_equal(_E2M1[idx], mag)
    nib = np.where(code_val < 0, idx | 8, idx).astype(np.uint8)
    sidx = np.searchsorted(_E4M3, sb)
    assert np.array_equal(_E4M3[sidx], sb)
    return nib, sidx.astype(np.uint8)


def unpack(codes: np.ndarray) -> np.ndarray:
    """[rows, K/2] bytes -> [rows, K] nibbles, element 2j in the low nibble of byte j."""
    out = np.empty((codes.shape[0], codes.shape[1] * 2), np.uint8)
    out[:, 0::2] = codes & 15
    out[:, 1::2] = codes >> 4
    return out


def check_act(spec, layer, x, T):
    r = layer.nvfp4_act(T)
    ent = layer.routing(T)["entries"]
    tok = ent // spec.top_k
    oracle_x = Layer.from_spec(spec, {}).widen_x(x).astype(np.float32)
    code_val, sb, ts = nvfp4_activation_parts(oracle_x)
    nib, sbytes = expected_bytes(code_val.reshape(T, -1), sb)
    got_nib = unpack(r["codes"])
    want_nib = nib[tok]
    # a zero code may carry either sign bit
    same = (got_nib == want_nib) | (((got_nib & 7) == 0) & ((want_nib & 7) == 0))
    bad = np.argwhere(~same)
    assert bad.size == 0, f"{len(bad)} codes differ, first (row, col) {bad[:4].tolist()}"
    assert np.array_equal(r["scales"], sbytes[tok]), "E4M3 block scales differ"
    assert np.float32(r["amax"][0]) / np.float32(2688.0) == ts


_cache = {}


def small_nvfp4():
    import quantized_moe_noaux_b300 as moe
    if "l" not in _cache:
        spec = LAYERS["small_nvfp4"]
        arrays = make_layer(spec)
        _cache["l"] = (spec, arrays, moe.MoeLayer.from_spec(spec, arrays, max_tokens=512))
    return _cache["l"]


@pytest.mark.parametrize("T,step", [(1, 11), (37, 12), (300, 13)])
def test_nvfp4_act_bytes_small(T, step):
    import quantized_moe_noaux_b300 as moe
    spec, _, layer = small_nvfp4()
    layer.set_path(moe.PATH_GROUPED)
    x = make_x(spec, T, step)
    out = empty_out(T, spec.hidden, spec.act_dtype)
    layer.forward(x_to_device(x, spec.act_dtype), out)
    torch.cuda.synchronize()
    assert layer.status() == 0
    check_act(spec, layer, x, T)
    layer.set_path(moe.PATH_AUTO)


def test_nvfp4_zero_activations():
    import quantized_moe_noaux_b300 as moe
    spec, arrays, layer = small_nvfp4()
    layer.set_path(moe.PATH_GROUPED)
    T = 5
    x = np.zeros((T, spec.hidden), np.uint16 if spec.act_dtype == "bf16" else np.float32)
    out = empty_out(T, spec.hidden, spec.act_dtype)
    layer.forward(x_to_device(x, spec.act_dtype), out)
    torch.cuda.synchronize()
    assert layer.status() == 0
    r = layer.nvfp4_act(T)
    assert not r["codes"].any() and not r["scales"].any() and r["amax"][0] == 0
    ref = Layer.from_spec(spec, arrays).forward(x)
    check_out(ref.out, out_to_host(out))
    assert not out_to_host(out).any()
    layer.set_path(moe.PATH_AUTO)
