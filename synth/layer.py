"""Seeded synthetic inputs for the quantised routed-MoE layer.

This module draws every input the layer consumes and nothing else:

* the router matrix ``W_r[E, H]`` ~ N(0, 1/H) (fp32, or rounded to bf16),
* the selection bias ``e_score_correction_bias[E]`` ~ N(0, bias_std),
* each expert's SwiGLU weights ``W_gu[2I, H]`` (rows 0..I-1 gate, I..2I-1 up) and
  ``W_d[H, I]``, drawn fp32 ~ N(0, 0.02) and stored in the format the layer reads
  (int4 with an fp16 scale per 32 input-dim elements, NVFP4, or bf16),
* the token activations ``x[T, H]`` ~ N(0, 1) (fp32, or rounded to bf16).

Storing drawn fp32 weights in a quantised container is the job of an offline
converter on the pages (colibri's FP8-to-int4 converter in "Show HN: Menjalankan GLM 5.2
di komputer lambat", section "Fitur utama yang diimplementasikan"; NVIDIA's Model
Optimizer in "NVIDIA stellt neues GLM-5.2 NVFP4 Modell vor", section "Technische
Details und Quantisierungsansatz"). It is input preparation here, not part of the
layer's forward pass: the router, the dequantisation, SwiGLU and the combine live in
the oracle and in the CUDA library, each written separately, and both take this
module's arrays as inputs.

Random streams (numpy ``default_rng`` over a ``SeedSequence``):

* ``[seed, 0]``: ``W_r`` (standard normal fp32, times 1/sqrt(H)),
* ``[seed, 1]``: the bias (standard normal fp32, times bias_std),
* ``[seed, 2, e]``: expert ``e`` (routed 0..E-1, the shared expert is ``e = E``):
  ``W_gu`` then ``W_d``, standard normal fp32 times 0.02,
* ``1000 + step``: ``x`` of that step (standard normal fp32).

One stream per expert lets a process pool draw a 257-expert layer in parallel while
staying bit-identical to a serial draw.
"""

from __future__ import annotations

import functools
import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor
from dataclasses import dataclass, replace

import numpy as np

__all__ = [
    "LayerSpec", "Workload", "LAYERS", "WORKLOADS", "make_layer", "make_router", "make_x",
    "f32_to_bf16_bits", "bf16_bits_to_f32", "quantize_int4_g32", "quantize_nvfp4_weight",
]


# ----------------------------------------------------------------------------- specs

@dataclass(frozen=True)
class LayerSpec:
    """Shape and storage formats of one MoE layer."""

    name: str
    hidden: int            # H
    inter: int             # I (per-expert intermediate size)
    n_experts: int         # E routed experts (plus one shared expert)
    top_k: int
    n_group: int
    topk_group: int
    rsf: float             # routed_scaling_factor
    weight_format: str     # "int4_g32" | "nvfp4"  (routed experts)
    act_dtype: str         # "f32" | "bf16"        (x and out)
    router_dtype: str      # "f32" | "bf16"
    shared_format: str     # "int4_g32" | "bf16"
    bias_std: float
    seed: int = 0
    weight_std: float = 0.02
    expert_top_p: float = 0.0  # adaptive expert top-p (0 = off)
    act_quant: str = "none"    # "none" | "q8_0" (int8 activations into the expert matmuls)

    @property
    def experts_per_group(self) -> int:
        return self.n_experts // self.n_group


@dataclass(frozen=True)
class Workload:
    """One layer run on ``tokens`` tokens per step for ``steps`` steps."""

    name: str
    layer: LayerSpec
    tokens: int
    steps: int = 1


_TINY = LayerSpec("tiny_h256_e16", hidden=256, inter=128, n_experts=16, top_k=4, n_group=4,
                  topk_group=2, rsf=2.5, weight_format="int4_g32", act_dtype="f32",
                  router_dtype="f32", shared_format="int4_g32", bias_std=0.01)
_GLM = LayerSpec("glm52_h6144_e256_int4g32", hidden=6144, inter=2048, n_experts=256, top_k=8,
                 n_group=8, topk_group=4, rsf=2.5, weight_format="int4_g32", act_dtype="bf16",
                 router_dtype="f32", shared_format="int4_g32", bias_std=0.01)

_SMALL = LayerSpec("small_h2048_e32", hidden=2048, inter=2048, n_experts=32, top_k=4, n_group=4,
                   topk_group=2, rsf=2.5, weight_format="int4_g32", act_dtype="bf16",
                   router_dtype="f32", shared_format="int4_g32", bias_std=0.01)

LAYERS = {
    "tiny": _TINY,
    # smallest shape the fused decode kernel runs (2048-column panels, 32-expert groups)
    "small": _SMALL,
    # the same shape with NVFP4 routed experts, bf16 router and bf16 shared expert
    "small_nvfp4": replace(_SMALL, name="small_h2048_e32_nvfp4", weight_format="nvfp4",
                           router_dtype="bf16", shared_format="bf16"),
    "glm52": _GLM,
    # decode at T=4 / T=32: the router is left unbiased so tokens share experts
    "glm52_unbiased": replace(_GLM, name="glm52_h6144_e256_int4g32_bias0", bias_std=0.0),
    # prefill: a wide bias skews the per-expert load
    "glm52_skewed": replace(_GLM, name="glm52_h6144_e256_int4g32_bias0.5", bias_std=0.5),
    # GLM shapes with 64 routed experts and a wide bias: a 2.8 GB profiling stand-in for the
    # skewed prefill layer (same per-expert matrices, a quarter of the experts)
    "glm52_e64_skewed": replace(_GLM, name="glm52_h6144_e64_int4g32_bias0.5", n_experts=64,
                                bias_std=0.5),
    # NVFP4 routed experts; router and shared expert stay bf16
    "glm52_nvfp4": replace(_GLM, name="glm52_h6144_e256_nvfp4", weight_format="nvfp4",
                           router_dtype="bf16", shared_format="bf16"),
    # adaptive expert top-p 0.7 (the pages' --topp 0.7) on the same weights
    "small_topp": replace(_SMALL, expert_top_p=0.7),
    "small_nvfp4_topp": replace(_SMALL, name="small_h2048_e32_nvfp4", weight_format="nvfp4",
                                router_dtype="bf16", shared_format="bf16", expert_top_p=0.7),
    "glm52_topp": replace(_GLM, expert_top_p=0.7),
    # the pages' per-row formats (scale per row; int8, packed int4, packed int2), and int4
    # per row with Q8_0-style int8 activations
    "small_int8_row": replace(_SMALL, name="small_h2048_e32_int8row", weight_format="int8_row",
                              shared_format="int8_row"),
    "small_int4_row": replace(_SMALL, name="small_h2048_e32_int4row", weight_format="int4_row",
                              shared_format="int4_row"),
    "small_int2_row": replace(_SMALL, name="small_h2048_e32_int2row", weight_format="int2_row",
                              shared_format="int2_row"),
    "small_int4_row_q8": replace(_SMALL, name="small_h2048_e32_int4row", weight_format="int4_row",
                                 shared_format="int4_row", act_quant="q8_0"),
    # GLM-shaped NVFP4 with 64 routed experts: a 1.4 GB profiling stand-in of the NVFP4 layer
    "glm52_e64_nvfp4": replace(_GLM, name="glm52_h6144_e64_nvfp4", n_experts=64, weight_format="nvfp4",
                               router_dtype="bf16", shared_format="bf16"),
    # GLM expert shapes with 64 routed experts, one per weight format (per-format GEMV
    # comparison at T = 1)
    "glm52_e64_int4_g32": replace(_GLM, name="glm52_h6144_e64_int4g32", n_experts=64),
    "glm52_e64_int8_row": replace(_GLM, name="glm52_h6144_e64_int8row", n_experts=64,
                                  weight_format="int8_row", shared_format="int8_row"),
    "glm52_e64_int4_row": replace(_GLM, name="glm52_h6144_e64_int4row", n_experts=64,
                                  weight_format="int4_row", shared_format="int4_row"),
    "glm52_e64_int2_row": replace(_GLM, name="glm52_h6144_e64_int2row", n_experts=64,
                                  weight_format="int2_row", shared_format="int2_row"),
}

WORKLOADS = {
    "tiny_t4": Workload("tiny_t4", LAYERS["tiny"], tokens=4),
    "glm52_decode_t1": Workload("glm52_decode_t1", LAYERS["glm52"], tokens=1, steps=1000),
    "glm52_decode_t1_topp07": Workload("glm52_decode_t1_topp07", LAYERS["glm52_topp"], tokens=1, steps=1000),
    # MTP draft-verify: one forward over the accepted position and DRAFT draft positions of a
    # sequence (DRAFT = 2 and 4), batch-union over their experts; positions drawn
    # independently (the pages give no statistics of how their routing overlaps)
    "glm52_mtp_verify_t3": Workload("glm52_mtp_verify_t3", LAYERS["glm52"], tokens=3, steps=1000),
    "glm52_mtp_verify_t5": Workload("glm52_mtp_verify_t5", LAYERS["glm52"], tokens=5, steps=1000),
    # host-resident experts with an HBM cache per layer: decode through a stack of layers
    "glm52_hostcache_t1": Workload("glm52_hostcache_t1", LAYERS["glm52"], tokens=1, steps=48),
    # per-format GEMV comparison, T = 1 (E = 64 stand-in of the GLM layer)
    "glm52_e64_int4_g32_t1": Workload("glm52_e64_int4_g32_t1", LAYERS["glm52_e64_int4_g32"], tokens=1, steps=200),
    "glm52_e64_int8_row_t1": Workload("glm52_e64_int8_row_t1", LAYERS["glm52_e64_int8_row"], tokens=1, steps=200),
    "glm52_e64_int4_row_t1": Workload("glm52_e64_int4_row_t1", LAYERS["glm52_e64_int4_row"], tokens=1, steps=200),
    "glm52_e64_int2_row_t1": Workload("glm52_e64_int2_row_t1", LAYERS["glm52_e64_int2_row"], tokens=1, steps=200),
    "glm52_decode_t4": Workload("glm52_decode_t4", LAYERS["glm52_unbiased"], tokens=4),
    "glm52_decode_t32": Workload("glm52_decode_t32", LAYERS["glm52_unbiased"], tokens=32),
    "glm52_prefill_t2048": Workload("glm52_prefill_t2048", LAYERS["glm52_skewed"], tokens=2048),
    "glm52_nvfp4_t256": Workload("glm52_nvfp4_t256", LAYERS["glm52_nvfp4"], tokens=256),
    "glm52_nvfp4_t4096": Workload("glm52_nvfp4_t4096", LAYERS["glm52_nvfp4"], tokens=4096),
}


# ------------------------------------------------------------------- bf16 storage

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even); returns the uint16 bit pattern."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ------------------------------------------------------------ container encoders
# Offline-converter side: fp32 weights -> stored codes. Written independently of the
# oracle's decoders, which the oracle's tests check these encoders against.

def quantize_int4_g32(w: np.ndarray):
    """Symmetric int4 with one fp16 scale per 32 consecutive input-dim elements.

    scale = fp16_rne(float32(absmax(group)) / 7); code = clamp(rint_even(w / scale), -8, 7);
    a group whose scale is zero stores zero codes. Codes are two's-complement nibbles,
    element 2j in the low nibble and 2j+1 in the high nibble of byte j.
    Returns (codes uint8 [N, K/2], scales float16 [N, K/32]).
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    assert k % 32 == 0
    g = w.reshape(n, k // 32, 32)
    amax = np.max(np.abs(g), axis=2)
    scale = (amax / np.float32(7.0)).astype(np.float16)
    sf = scale.astype(np.float32)[..., None]
    q = np.zeros_like(g)
    np.divide(g, sf, out=q, where=sf != 0)
    q = np.clip(np.rint(q), -8, 7).astype(np.int8)
    u = (q.view(np.uint8) & np.uint8(0x0F)).reshape(n, k // 2, 2)
    codes = (u[..., 0] | (u[..., 1] << np.uint8(4))).astype(np.uint8)
    return codes, scale


def quantize_int_row(w: np.ndarray, bits: int):
    """Symmetric per-row integers (int8, packed int4, packed int2 with one scale per row).

    qmax = 2^(bits-1) - 1; scale = float32(absmax(row)) / qmax in fp32; code =
    clamp(rint_even(w / scale), -qmax - 1, qmax) (a zero row stores zero codes). Packing:
    int8 one per byte; int4 element 2j in the low nibble of byte j; int2 element 4j + i in
    bits 2i..2i+1 of byte j (two's complement fields).
    Returns (codes uint8 [N, K * bits / 8], scales float32 [N, 1]).
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    per = 8 // bits
    assert k % per == 0
    qmax = (1 << (bits - 1)) - 1
    scale = (np.max(np.abs(w), axis=1) / np.float32(qmax)).astype(np.float32)
    q = np.zeros_like(w)
    np.divide(w, scale[:, None], out=q, where=scale[:, None] != 0)
    q = np.clip(np.rint(q), -qmax - 1, qmax).astype(np.int64)
    u = (q & ((1 << bits) - 1)).reshape(n, k // per, per)
    codes = np.zeros((n, k // per), np.int64)
    for i in range(per):
        codes |= u[..., i] << (bits * i)
    return codes.astype(np.uint8), scale.reshape(n, 1)


_ROW_BITS = {"int8_row": 8, "int4_row": 4, "int2_row": 2}


def _grid_e4m3() -> np.ndarray:
    """Magnitudes of the 127 finite non-negative E4M3 codes 0x00..0x7E, by code."""
    c = np.arange(127)
    e, m = c >> 3, c & 7
    return np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))


def _grid_e2m1() -> np.ndarray:
    """Magnitudes of the 8 non-negative E2M1 codes 0..7, by code."""
    c = np.arange(8)
    e, m = c >> 1, c & 1
    return np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * 2.0 ** (e - 1.0))


def _round_to_grid(mag: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Code of the grid value nearest to ``mag`` (>= 0); ties go to the even code;
    magnitudes beyond the largest grid value saturate to it."""
    mag = np.asarray(mag, dtype=np.float64)
    hi = np.clip(np.searchsorted(grid, mag, side="left"), 1, len(grid) - 1)
    lo = hi - 1
    dlo = mag - grid[lo]
    dhi = grid[hi] - mag
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    return np.where(mag >= grid[-1], len(grid) - 1, code).astype(np.uint8)


def quantize_nvfp4_weight(w: np.ndarray):
    """NVFP4 storage of one weight matrix: E2M1 codes, an E4M3 scale per 16 consecutive
    input-dim elements and one fp32 tensor scale.

    All arithmetic is fp32: tensor_scale = amax(|W|) / 2688 (6 * 448); block scale
    = e4m3_rne_satfinite(amax16 / 6 / tensor_scale); code = e2m1_rne_satfinite(w /
    (block_scale * tensor_scale)); zero divisors store zero codes.
    Returns (codes uint8 [N, K/2] low nibble = even element, scales uint8 [N, K/16]
    (E4M3 bit patterns), tensor_scale float32).
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    assert k % 16 == 0
    ts = np.float32(np.max(np.abs(w))) / np.float32(6.0 * 448.0)
    blocks = w.reshape(n, k // 16, 16)
    bamax = np.max(np.abs(blocks), axis=2)
    if ts == 0:
        sb_code = np.zeros(bamax.shape, np.uint8)
    else:
        sb_code = _round_to_grid((bamax / np.float32(6.0)) / ts, _grid_e4m3())
    sb = _grid_e4m3()[sb_code].astype(np.float32)
    denom = (sb * ts).astype(np.float32)[..., None]
    r = np.zeros_like(blocks)
    np.divide(blocks, denom, out=r, where=denom != 0)
    mag = _round_to_grid(np.abs(r), _grid_e2m1())
    code = np.where((r < 0) & (mag != 0), mag | np.uint8(8), mag).astype(np.uint8)
    code = code.reshape(n, k // 2, 2)
    packed = (code[..., 0] | (code[..., 1] << np.uint8(4))).astype(np.uint8)
    return packed, sb_code, np.float32(ts)


# ---------------------------------------------------------------------- drawing

def _expert_rng(seed: int, e: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed, 2, e]))


def _draw_expert(args):
    """Draw expert ``e`` and store it in ``fmt``; module level so a spawn pool can run it."""
    seed, e, hidden, inter, std, fmt = args
    rng = _expert_rng(seed, e)
    w_gu = rng.standard_normal((2 * inter, hidden), dtype=np.float32) * np.float32(std)
    w_d = rng.standard_normal((hidden, inter), dtype=np.float32) * np.float32(std)
    if fmt == "int4_g32":
        gc, gs = quantize_int4_g32(w_gu)
        dc, ds = quantize_int4_g32(w_d)
        return {"gu_codes": gc, "gu_scales": gs, "d_codes": dc, "d_scales": ds}
    if fmt == "nvfp4":
        gc, gs, gt = quantize_nvfp4_weight(w_gu)
        dc, ds, dt = quantize_nvfp4_weight(w_d)
        return {"gu_codes": gc, "gu_scales": gs, "gu_tscale": gt,
                "d_codes": dc, "d_scales": ds, "d_tscale": dt}
    if fmt == "bf16":
        return {"gu_bf16": f32_to_bf16_bits(w_gu), "d_bf16": f32_to_bf16_bits(w_d)}
    if fmt in _ROW_BITS:
        gc, gs = quantize_int_row(w_gu, _ROW_BITS[fmt])
        dc, ds = quantize_int_row(w_d, _ROW_BITS[fmt])
        return {"gu_codes": gc, "gu_scales": gs, "d_codes": dc, "d_scales": ds}
    raise ValueError(f"unknown weight format {fmt!r}")


def _alloc_expert_arrays(n: int, hidden: int, inter: int, fmt: str, prefix: str) -> dict:
    if fmt == "int4_g32":
        return {f"{prefix}gu_codes": np.empty((n, 2 * inter, hidden // 2), np.uint8),
                f"{prefix}gu_scales": np.empty((n, 2 * inter, hidden // 32), np.float16),
                f"{prefix}d_codes": np.empty((n, hidden, inter // 2), np.uint8),
                f"{prefix}d_scales": np.empty((n, hidden, inter // 32), np.float16)}
    if fmt == "nvfp4":
        return {f"{prefix}gu_codes": np.empty((n, 2 * inter, hidden // 2), np.uint8),
                f"{prefix}gu_scales": np.empty((n, 2 * inter, hidden // 16), np.uint8),
                f"{prefix}gu_tscale": np.empty((n,), np.float32),
                f"{prefix}d_codes": np.empty((n, hidden, inter // 2), np.uint8),
                f"{prefix}d_scales": np.empty((n, hidden, inter // 16), np.uint8),
                f"{prefix}d_tscale": np.empty((n,), np.float32)}
    if fmt == "bf16":
        return {f"{prefix}gu_bf16": np.empty((n, 2 * inter, hidden), np.uint16),
                f"{prefix}d_bf16": np.empty((n, hidden, inter), np.uint16)}
    if fmt in _ROW_BITS:
        per = 8 // _ROW_BITS[fmt]
        return {f"{prefix}gu_codes": np.empty((n, 2 * inter, hidden // per), np.uint8),
                f"{prefix}gu_scales": np.empty((n, 2 * inter, 1), np.float32),
                f"{prefix}d_codes": np.empty((n, hidden, inter // per), np.uint8),
                f"{prefix}d_scales": np.empty((n, hidden, 1), np.float32)}
    raise ValueError(fmt)


def _default_workers(n_items: int, hidden: int) -> int:
    if hidden * n_items < 1 << 20:
        return 0
    return max(1, min(os.cpu_count() or 1, 64, n_items))


def make_router(spec: LayerSpec):
    """The router matrix and the selection bias of ``spec`` (the same arrays
    ``make_layer`` returns; both come from streams independent of the experts)."""
    H, E = spec.hidden, spec.n_experts
    rng_r = np.random.default_rng(np.random.SeedSequence([spec.seed, 0]))
    wr = rng_r.standard_normal((E, H), dtype=np.float32) * np.float32(1.0 / np.sqrt(H))
    wr = f32_to_bf16_bits(wr) if spec.router_dtype == "bf16" else wr
    rng_b = np.random.default_rng(np.random.SeedSequence([spec.seed, 1]))
    bias = rng_b.standard_normal(E, dtype=np.float32) * np.float32(spec.bias_std)
    return wr, bias


@functools.lru_cache(maxsize=2)
def make_layer(spec: LayerSpec, workers: int | None = None) -> dict:
    """Draw one layer. Returns read-only numpy arrays:

    ``router_w`` [E, H] (float32, or uint16 bf16 bits), ``bias`` [E] float32,
    routed experts ``gu_codes`` [E, 2I, H/2] uint8, ``gu_scales`` [E, 2I, H/32] float16
    (int4_g32) or [E, 2I, H/16] uint8 E4M3 (nvfp4), ``d_codes`` [E, H, I/2],
    ``d_scales`` [E, H, I/32 | I/16], nvfp4 only: ``gu_tscale`` / ``d_tscale`` [E] float32;
    the shared expert under the ``sh_`` prefix with a leading dimension of 1, either in
    the same int4/nvfp4 layout or as ``sh_gu_bf16`` [1, 2I, H] / ``sh_d_bf16`` [1, H, I].
    """
    H, I, E = spec.hidden, spec.inter, spec.n_experts
    assert H % 32 == 0 and I % 32 == 0 and E % spec.n_group == 0
    out: dict = {}
    out["router_w"], out["bias"] = make_router(spec)

    out.update(_alloc_expert_arrays(E, H, I, spec.weight_format, ""))
    out.update(_alloc_expert_arrays(1, H, I, spec.shared_format, "sh_"))
    jobs = [(spec.seed, e, H, I, spec.weight_std, spec.weight_format) for e in range(E)]
    jobs.append((spec.seed, E, H, I, spec.weight_std, spec.shared_format))

    def _store(e, res):
        prefix, row = ("", e) if e < E else ("sh_", 0)
        for key, val in res.items():
            out[prefix + key][row] = val

    nw = _default_workers(len(jobs), H) if workers is None else workers
    if nw <= 1:
        for job in jobs:
            _store(job[1], _draw_expert(job))
    else:
        with ProcessPoolExecutor(max_workers=nw, mp_context=mp.get_context("spawn")) as ex:
            for job, res in zip(jobs, ex.map(_draw_expert, jobs, chunksize=1)):
                _store(job[1], res)
    for val in out.values():
        val.flags.writeable = False
    return out


def with_bias_of(arrays: dict, spec: LayerSpec) -> dict:
    """``arrays`` (a layer drawn for a spec that differs from ``spec`` only in bias_std)
    with the bias of ``spec``: equal to ``make_layer(spec)`` without redrawing experts."""
    out = dict(arrays)
    out["bias"] = make_router(spec)[1]
    out["bias"].flags.writeable = False
    return out


def make_x(spec: LayerSpec, tokens: int, step: int = 0) -> np.ndarray:
    """Activations of one step, drawn with seed ``1000 + step``: float32 [T, H] for
    fp32 layers, uint16 bf16 bit patterns [T, H] for bf16 layers."""
    rng = np.random.default_rng(1000 + step)
    x = rng.standard_normal((tokens, spec.hidden), dtype=np.float32)
    return f32_to_bf16_bits(x) if spec.act_dtype == "bf16" else x
