"""Seeded synthetic inputs for the quantised routed-MoE layer (see ``synth.layer``)."""

from .layer import (  # noqa: F401
    LayerSpec,
    Workload,
    LAYERS,
    WORKLOADS,
    make_layer,
    make_router,
    with_bias_of,
    make_x,
    f32_to_bf16_bits,
    bf16_bits_to_f32,
    quantize_int4_g32,
    quantize_nvfp4_weight,
)
