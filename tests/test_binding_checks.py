"""The binding refuses activation buffers of the wrong shape, element type or memory kind
before calling the library (which cannot see them, and whose kernels would read or write
outside such a buffer or dereference a host address). A buffer that passes reaches the
library: with a NULL layer handle that call returns MOE_ERR_INVALID_ARG (CPU only; stream 0
is the legacy default stream, so no CUDA context is needed)."""

import numpy as np
import pytest
import torch

import quantized_moe_noaux_b300 as moe


def layer(act_dtype, hidden=256):
    L = object.__new__(moe.MoeLayer)      # no library object: the handle stays NULL
    L.hidden, L.act_dtype, L.top_k, L.n_experts = hidden, act_dtype, 4, 16
    L._h = moe._P()
    return L


def reaches_library(call):
    with pytest.raises(moe.MoeError) as ei:
        call()
    return ei.value.code == 1


def test_forward_host_accepts_host_buffers_of_the_layer_type():
    L = layer("f32")
    assert reaches_library(lambda: L.forward_host(np.zeros((3, 256), np.float32), np.zeros((3, 256), np.float32), 0))
    assert reaches_library(lambda: L.forward_host(torch.zeros(3, 256), torch.zeros(3, 256), 0))
    B = layer("bf16")
    assert reaches_library(lambda: B.forward_host(np.zeros((2, 256), np.uint16), np.zeros((2, 256), np.uint16), 0))
    assert reaches_library(lambda: B.forward_host(torch.zeros(2, 256, dtype=torch.bfloat16),
                                                  torch.zeros(2, 256, dtype=torch.bfloat16), 0))


@pytest.mark.parametrize("x,out,exc", [
    (np.zeros((3, 128), np.float32), np.zeros((3, 128), np.float32), ValueError),     # wrong H
    (np.zeros(256, np.float32), np.zeros(256, np.float32), ValueError),               # not 2-D
    (np.zeros((3, 256), np.float64), np.zeros((3, 256), np.float64), TypeError),      # wrong type
    (np.zeros((3, 256), np.float32), np.zeros((2, 256), np.float32), ValueError),     # row count
    ([[0.0] * 256], np.zeros((1, 256), np.float32), TypeError),                       # not an array
])
def test_forward_host_refusals(x, out, exc):
    with pytest.raises(exc):
        layer("f32").forward_host(x, out)


def test_bf16_layer_refuses_other_16_and_32_bit_types():
    B = layer("bf16")
    with pytest.raises(TypeError):
        B.forward_host(np.zeros((2, 256), np.float32), np.zeros((2, 256), np.float32))
    with pytest.raises(TypeError):
        B.forward_host(torch.zeros(2, 256, dtype=torch.float16), torch.zeros(2, 256, dtype=torch.float16))


def test_device_entry_points_refuse_host_memory():
    L = layer("f32")
    for bad in (np.zeros((3, 256), np.float32), torch.zeros(3, 256)):
        with pytest.raises(TypeError):
            L.forward(bad, bad)
        with pytest.raises(TypeError):
            L.prefetch(bad)


def test_trace_buffer_must_be_a_large_enough_device_tensor():
    L = layer("f32")
    with pytest.raises(TypeError):
        L.set_trace(torch.zeros((148, 64), dtype=torch.int64), 148)      # host memory
    with pytest.raises(TypeError):
        L.set_trace(np.zeros((148, 64), np.int64), 148)
    assert reaches_library(lambda: L.set_trace(None, 148))              # switching off


def test_weight_sizes_follow_the_header_layout_for_every_generated_layer():
    """weight_bytes (the header's layout table) against the arrays the generator allocates
    for every layer spec: its per-expert allocation (no data drawn) times E for the routed
    experts, once for the shared expert, and its router arrays."""
    from synth import LAYERS
    from synth.layer import _alloc_expert_arrays, make_router
    for name, s in LAYERS.items():
        want = moe.weight_bytes(s.hidden, s.inter, s.n_experts, s.weight_format, s.shared_format,
                                s.router_dtype)
        got = {k: moe._nbytes(a) * s.n_experts
               for k, a in _alloc_expert_arrays(1, s.hidden, s.inter, s.weight_format, "").items()}
        got.update({k: moe._nbytes(a)
                    for k, a in _alloc_expert_arrays(1, s.hidden, s.inter, s.shared_format, "sh_").items()})
        router_w, bias = make_router(s)
        got.update(router_w=router_w.nbytes, bias=bias.nbytes)
        assert got == want, (name, {k: (got.get(k), want.get(k)) for k in set(got) | set(want)
                                    if got.get(k) != want.get(k)})


def test_weight_arrays_of_the_wrong_size_are_refused_before_creation():
    from synth import LAYERS
    from synth.layer import make_layer
    spec = LAYERS["tiny"]
    arrays = make_layer(spec)
    short = dict(arrays, gu_scales=arrays["gu_scales"][:, :, :4].copy())      # scales per 64
    with pytest.raises(ValueError):
        moe.MoeLayer.from_spec(spec, short, max_tokens=4, stream=0)
    wide = dict(arrays, router_w=np.zeros((spec.n_experts, 2 * spec.hidden), np.float32))
    with pytest.raises(ValueError):
        moe.MoeLayer.from_spec(spec, wide, max_tokens=4, stream=0)
    # the right sizes reach the library (no device here: MOE_ERR_CUDA)
    with pytest.raises(moe.MoeError) as ei:
        moe.MoeLayer.from_spec(spec, arrays, max_tokens=4, stream=0)
    assert ei.value.code == 4


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without libmoe.so every use of the library raises; there is no fallback path."""
    monkeypatch.setattr(moe, "LIB_PATH", str(tmp_path / "libmoe.so"))
    monkeypatch.setattr(moe, "_lib", None)
    with pytest.raises(ImportError, match="no fallback"):
        moe.lib
    with pytest.raises(ImportError):
        layer("f32").forward_host(np.zeros((1, 256), np.float32), np.zeros((1, 256), np.float32), 0)
