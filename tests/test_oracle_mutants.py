"""Planted mistakes in the oracle must be caught by its pins.

Each mutant replaces one oracle function with a plausible wrong variant (a dropped
term, a wrong sign or index, a transposed operand, a wrong tie rule) for the duration
of one test, on the CPU, and asserts that at least one pin fails.
"""

import numpy as np
import pytest

from oracle import moe_oracle as O
from tests import oracle_pins as P

_orig = {name: getattr(O, name) for name in dir(O)}


def _nibbles_swapped(codes):
    v = _orig["decode_int4"](codes)
    out = v.copy()
    out[..., 0::2], out[..., 1::2] = v[..., 1::2], v[..., 0::2]
    return out


def _unsigned_int4(codes):
    v = _orig["decode_int4"](codes)
    return np.where(v < 0, v + 16, v)


def _scale_group_shift(codes, scales):
    return _orig["dequant_int4_g32"](codes, np.roll(np.asarray(scales), 1, axis=-1))


def _e4m3_bias8(bits):
    return _orig["decode_e4m3"](bits) / 2.0


def _e2m1_subnormal(n):
    v = _orig["decode_e2m1"](n)
    return np.where(np.abs(v) == 0.5, v / 2, v)


def _sigmoid_sign(z):
    return 1.0 / (1.0 + np.exp(z))


def _silu_sign(z):
    return z / (1.0 + np.exp(z))


def _swiglu_swapped(w_gu, xr):
    gu = np.asarray(xr, np.float64) @ np.asarray(w_gu, np.float64).T
    i = gu.shape[1] // 2
    return O.silu(gu[:, i:]) * gu[:, :i]


def _down_transposed(w_d, h):
    return np.asarray(h, np.float64) @ np.asarray(w_d, np.float64)


def _select_top1_group(scores, bias, n_group, topk_group, top_k):
    # group score from the single largest b instead of the top-2 sum
    s = np.asarray(scores, np.float64)
    T, E = s.shape
    G = E // n_group
    b = s + np.asarray(bias)[None]
    ids = np.empty((T, top_k), np.int64)
    for t in range(T):
        gs = b[t].reshape(n_group, G).max(1)
        kept = np.argsort(-gs, kind="stable")[:topk_group]
        m = np.full(E, -np.inf)
        for g in kept:
            m[g * G:(g + 1) * G] = b[t, g * G:(g + 1) * G]
        ids[t] = np.argsort(-m, kind="stable")[:top_k]
    return O.Selection(ids, np.full(T, np.inf), np.full(T, np.inf))


def _select_zero_fill(scores, bias, n_group, topk_group, top_k):
    s = np.asarray(scores, np.float64)
    T, E = s.shape
    G = E // n_group
    b = s + np.asarray(bias)[None]
    ids = np.empty((T, top_k), np.int64)
    for t in range(T):
        grp = b[t].reshape(n_group, G)
        gs = np.sort(grp, 1)[:, -2:].sum(1)
        kept = np.argsort(-gs, kind="stable")[:topk_group]
        m = np.zeros(E)
        for g in kept:
            m[g * G:(g + 1) * G] = b[t, g * G:(g + 1) * G]
        ids[t] = np.argsort(-m, kind="stable")[:top_k]
    return O.Selection(ids, np.full(T, np.inf), np.full(T, np.inf))


def _select_ties_high(scores, bias, n_group, topk_group, top_k):
    # mirror the expert axis so equal scores resolve to the higher index
    E = np.asarray(scores).shape[1]
    sel = _orig["select_experts"](np.asarray(scores)[:, ::-1], np.asarray(bias)[::-1],
                                  n_group, topk_group, top_k)
    return O.Selection(E - 1 - sel.ids, sel.group_margin, sel.expert_margin)


def _select_bias_ignored(scores, bias, n_group, topk_group, top_k):
    return _orig["select_experts"](scores, np.zeros_like(np.asarray(bias)), n_group,
                                   topk_group, top_k)


def _weights_no_rsf(scores, ids, rsf):
    return _orig["routing_weights"](scores, ids, 1.0)


def _weights_unnormalised(scores, ids, rsf):
    return np.take_along_axis(np.asarray(scores, np.float64), ids, axis=1) * rsf


def _group_descending(ids, n_experts):
    counts, offsets, lst = _orig["group_tokens"](ids, n_experts)
    lst = lst.copy()
    for e in range(n_experts):
        lst[offsets[e]:offsets[e + 1]] = lst[offsets[e]:offsets[e + 1]][::-1]
    return counts, offsets, lst


def _act_scale_no6(a):
    a32 = np.asarray(a, np.float32)
    return _orig["quantize_nvfp4_activation"](a32 * np.float32(6.0)) / 6.0 * 1.0001


def _h_scale_per_expert(hs):
    # each routed expert's h rows quantised with a tensor scale of their own
    return {e: (ent, _orig["quantize_nvfp4_activation"](np.asarray(h, np.float32))) for e, (ent, h) in hs.items()}


def _shared_reads_quantised_x(shared_format, x64, x_in):
    return x_in


def _widen_bf16_truncating(bits):
    # drops the lowest mantissa bit of every pattern
    return _orig["widen_bf16"](np.asarray(bits, np.uint16) & np.uint16(0xFFFE))


def _top_p_variant(scores, ids, p, le=False, slot_order=False, ties_high=False):
    s = np.asarray(scores, np.float64)
    ids = np.asarray(ids, np.int64)
    keep = np.ones(ids.shape, bool)
    if not 0.0 < p < 1.0:
        return O.TopP(keep, np.full(ids.shape[0], np.inf))
    for t in range(ids.shape[0]):
        sel = s[t, ids[t]]
        if slot_order:
            order = np.arange(ids.shape[1])
        else:
            order = np.lexsort((-ids[t] if ties_high else ids[t], -sel))
        before = np.concatenate([[0.0], np.cumsum(sel[order])[:-1]])
        keep[t, order] = before <= p * sel.sum() if le else before < p * sel.sum()
    return O.TopP(keep, np.full(ids.shape[0], np.inf))


def _weights_dropped_unmasked(scores, ids, rsf):
    # forgets that -1 marks a dropped slot (indexes the last expert instead)
    sel = np.take_along_axis(np.asarray(scores, np.float64), np.asarray(ids), axis=1)
    return sel / sel.sum(axis=1, keepdims=True) * rsf


def _group_dropped_counted(ids, n_experts):
    return _orig["group_tokens"](np.asarray(ids) % n_experts, n_experts)


def _int_row_fields_reversed(codes, bits):
    v = _orig["decode_int_row"](codes, bits)
    per = 8 // bits
    return v.reshape(v.shape[:-1] + (-1, per))[..., ::-1].reshape(v.shape)


def _int_row_unsigned(codes, bits):
    v = _orig["decode_int_row"](codes, bits)
    return np.where(v < 0, v + (1 << bits), v)


def _q8_0_no_fp16_step(a):
    a32 = np.asarray(a, np.float32)
    m, k = a32.shape
    blk = a32.reshape(m, k // 32, 32)
    d = (np.max(np.abs(blk), axis=2) / np.float32(127.0)).astype(np.float32)
    q = np.zeros(blk.shape, np.float32)
    np.divide(blk, d[..., None], out=q, where=d[..., None] != 0)
    return (np.clip(np.rint(q), -127, 127) * d[..., None]).astype(np.float64).reshape(m, k)


def _q8_0_round_half_up(a):
    a32 = np.asarray(a, np.float32)
    m, k = a32.shape
    blk = a32.reshape(m, k // 32, 32)
    d = (np.max(np.abs(blk), axis=2) / np.float32(127.0)).astype(np.float16).astype(np.float32)
    q = np.zeros(blk.shape, np.float32)
    np.divide(blk, d[..., None], out=q, where=d[..., None] != 0)
    q = np.sign(q) * np.floor(np.abs(q) + 0.5)
    return (np.clip(q, -127, 127) * d[..., None]).astype(np.float64).reshape(m, k)


def _q8_0_h_unquantised(a):
    # a wiring mistake of the layer: its h step (the `hidden` wrapper inside Layer.forward)
    # skips the quantisation; every other caller gets the real quantiser
    import sys
    if sys._getframe(1).f_code.co_name == "hidden":
        return np.asarray(a, np.float64)
    return _orig["quantize_q8_0_activation"](a)


def _select_variant(kind):
    """noaux_tc selection with one step changed: the group score summed over the whole
    group, no group mask, or groups ranked by the unbiased scores."""
    def select(scores, bias, n_group, topk_group, top_k):
        s = np.asarray(scores, np.float64)
        T, E = s.shape
        G = E // n_group
        b = s + np.asarray(bias)[None]
        ids = np.empty((T, top_k), np.int64)
        for t in range(T):
            grp = (s[t] if kind == "groups_unbiased" else b[t]).reshape(n_group, G)
            gs = grp.sum(1) if kind == "group_sum_all" else np.sort(grp, 1)[:, -2:].sum(1)
            kept = np.argsort(-gs, kind="stable")[:topk_group]
            m = b[t].copy() if kind == "no_group_mask" else np.full(E, -np.inf)
            if kind != "no_group_mask":
                for g in kept:
                    m[g * G:(g + 1) * G] = b[t, g * G:(g + 1) * G]
            ids[t] = np.argsort(-m, kind="stable")[:top_k]
        return O.Selection(ids, np.full(T, np.inf), np.full(T, np.inf))
    return select


def _softmax(z):
    z = np.asarray(z, np.float64)
    e = np.exp(z - z.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def _weights_slot_rolled(scores, ids, rsf):
    return np.roll(_orig["routing_weights"](scores, ids, rsf), 1, axis=1)


def _silu_without_x(z):
    return 1.0 / (1.0 + np.exp(-np.asarray(z, np.float64)))


def _widen_as_fp16(bits):
    return np.asarray(bits).astype(np.uint16).view(np.float16).astype(np.float64)


def _e4m3_no_subnormal(bits):
    # exponent field 0 read as a normal number (implicit leading 1)
    b = np.asarray(bits).astype(np.int64)
    exp, man = (b >> 3) & 15, b & 7
    sgn = np.where(b & 128, -1.0, 1.0)
    return np.where(exp == 0, sgn * (1 + man / 8.0) * 2.0 ** -6, _orig["decode_e4m3"](bits))


def _e2m1_sign_ignored(n):
    return np.abs(_orig["decode_e2m1"](n))


def _q8_0_block16(a):
    # blocks of 16 elements instead of 32
    a = np.asarray(a, np.float64)
    out = np.empty_like(a).reshape(-1, 16)
    for i, blk in enumerate(a.reshape(-1, 16)):
        out[i] = _orig["quantize_q8_0_activation"](np.concatenate([blk, np.zeros(16)])[None])[0, :16]
    return out.reshape(a.shape)


def _int_row_scale_ignored(codes, scales, bits):
    return O.decode_int_row(codes, bits).astype(np.float64)


def _group_slot_major(ids, n_experts):
    counts, offsets, lst = _orig["group_tokens"](ids, n_experts)
    lst = lst.copy()
    k = np.shape(ids)[1]
    for e in range(n_experts):
        seg = lst[offsets[e]:offsets[e + 1]]
        lst[offsets[e]:offsets[e + 1]] = sorted(seg, key=lambda r: (r % k, r // k))
    return counts, offsets, lst


def _code_ties_away(mag, table):
    # nearest table entry, halfway cases away from zero instead of to the even entry
    mag = np.asarray(mag, np.float64)
    j = np.clip(np.searchsorted(table, mag, side="right") - 1, 0, len(table) - 2)
    up = (table[j + 1] - mag) <= (mag - table[j])
    return np.where(mag >= table[-1], len(table) - 1, j + up).astype(np.int64)


def _code_truncated(mag, table):
    mag = np.asarray(mag, np.float64)
    return np.clip(np.searchsorted(table, mag, side="right") - 1, 0, len(table) - 1).astype(np.int64)


def _nvfp4_parts_variant(kind):
    """NVFP4 activation quantiser with one step changed: E2M1 ties away from zero, E4M3
    block scales truncated, a tensor scale per row, block amax over 32 elements, or a
    tensor scale amax / 448."""
    def parts(a):
        a32 = np.asarray(a, np.float32)
        m, k = a32.shape
        if kind == "ts_per_row":
            amax = np.max(np.abs(a32), axis=1, keepdims=True).astype(np.float32)
        else:
            amax = np.float32(np.max(np.abs(a32)))
        den = np.float32(448.0 if kind == "ts_no6" else 2688.0)
        ts = (amax / den).astype(np.float32)
        if np.all(ts == 0):
            return np.zeros((m, k // 16, 16)), np.zeros((m, k // 16)), np.float32(0)
        blocks = a32.reshape(m, k // 16, 16)
        if kind == "amax32":
            bamax = np.repeat(np.max(np.abs(a32.reshape(m, k // 32, 32)), axis=2), 2, axis=1)
        else:
            bamax = np.max(np.abs(blocks), axis=2)
        ratio = ((bamax / np.float32(6.0)).astype(np.float32) / ts).astype(np.float32)
        scode = _code_truncated if kind == "e4m3_truncated" else O._rne_code
        sb = O._E4M3_MAGS[scode(ratio, O._E4M3_MAGS)]
        denom = (sb.astype(np.float32) * ts).astype(np.float32)
        q = np.zeros(blocks.shape, np.float32)
        np.divide(blocks, denom[..., None], out=q, where=denom[..., None] != 0)
        ecode = _code_ties_away if kind == "e2m1_ties_away" else O._rne_code
        vals = np.sign(q) * O._E2M1_MAGS[ecode(np.abs(q), O._E2M1_MAGS)]
        if kind == "ts_per_row":
            return vals, sb * ts, np.float32(1.0)
        return vals, sb, np.float32(ts)
    return parts


def _nvfp4_tensor_scale_ignored(codes, scales, tensor_scale):
    return _orig["dequant_nvfp4"](codes, scales, 1.0)


def _nvfp4_scale_per_32(codes, scales, tensor_scale):
    sc = np.asarray(scales, np.uint8)
    return _orig["dequant_nvfp4"](codes, np.repeat(sc[:, 0::2], 2, axis=1)[:, :sc.shape[1]], tensor_scale)


def _e4m3_no_nan(bits):
    # S.1111.111 read as +-480 instead of NaN
    b = np.asarray(bits).astype(np.int64) & 0xFF
    return np.where((b & 0x7F) == 0x7F, np.where(b & 0x80, -480.0, 480.0), _orig["decode_e4m3"](bits))


def _int4_scale_per_16(codes, scales):
    c = O.decode_int4(codes).astype(np.float64)
    sc = np.asarray(scales, np.float64)
    return c * sc[:, np.minimum(np.arange(c.shape[1]) // 16, sc.shape[1] - 1)]


def _q8_0_divide_by_128(a):
    a32 = np.asarray(a, np.float32)
    m, k = a32.shape
    blocks = a32.reshape(m, k // 32, 32)
    d = (np.max(np.abs(blocks), axis=2) / np.float32(128.0)).astype(np.float16).astype(np.float32)
    q = np.zeros(blocks.shape, np.float32)
    np.divide(blocks, d[..., None], out=q, where=d[..., None] != 0)
    return (np.clip(np.rint(q), -127, 127).astype(np.float64) * d[..., None]).reshape(m, k)


def _top_p_rule_variant(kind):
    """Adaptive top-p with one step changed: the threshold taken from the mass of all E
    experts, the expert that crosses the threshold dropped, or the experts ranked by id."""
    def top_p(scores, ids, p):
        ref = _orig["expert_top_p"](scores, ids, p)
        if not 0.0 < p < 1.0:
            return ref
        s = np.asarray(scores, np.float64)
        ids = np.asarray(ids, np.int64)
        keep = np.ones(ids.shape, bool)
        for t in range(ids.shape[0]):
            sel = s[t, ids[t]]
            order = np.argsort(ids[t]) if kind == "order_by_id" else np.lexsort((ids[t], -sel))
            ranked = sel[order]
            total = s[t].sum() if kind == "mass_of_all_E" else ranked.sum()
            upto = np.cumsum(ranked)
            before = np.concatenate([[0.0], upto[:-1]])
            kept = upto < p * total if kind == "crossing_dropped" else before < p * total
            kept[0] = True
            keep[t, order] = kept
        return O.TopP(keep, ref.margin)
    return top_p


def _top_p_margin_zero(scores, ids, p):
    r = _orig["expert_top_p"](scores, ids, p)
    return O.TopP(r.keep, np.where(np.isfinite(r.margin), 0.0, r.margin))


def _select_margins(value):
    def select(scores, bias, n_group, topk_group, top_k):
        r = _orig["select_experts"](scores, bias, n_group, topk_group, top_k)
        return O.Selection(r.ids, np.full_like(r.group_margin, value), np.full_like(r.expert_margin, value))
    return select


def _router_fp32(x, router_w):
    return (np.asarray(x, np.float32) @ np.asarray(router_w, np.float32).T).astype(np.float64)


def _sigmoid_fp32(z):
    z = np.asarray(z, np.float32)
    return (np.float32(1) / (np.float32(1) + np.exp(-z))).astype(np.float64)


def _silu_fp32(z):
    z = np.asarray(z, np.float32)
    return (z / (np.float32(1) + np.exp(-z))).astype(np.float64)


def _group_token_only(ids, n_experts):
    counts, offsets, lst = _orig["group_tokens"](ids, n_experts)
    return counts, offsets, lst // np.shape(ids)[1]


def _identity_glu_up_only(w_gu, xr):
    gu = np.asarray(xr, np.float64) @ np.asarray(w_gu, np.float64).T
    return gu[:, gu.shape[1] // 2:]


def _called_from_layer_forward():
    import sys
    return sys._getframe(2).f_code.co_name == "forward"


def _nvfp4_x_unquantised_in_layer(a):
    # wiring mistake: Layer.forward feeds the routed experts the unquantised x
    if _called_from_layer_forward():
        return np.asarray(a, np.float64)
    return _orig["quantize_nvfp4_activation"](a)


def _nvfp4_x_per_token_in_layer(a):
    # wiring mistake: Layer.forward quantises each token with a tensor scale of its own
    if _called_from_layer_forward():
        a = np.asarray(a)
        return np.vstack([_orig["quantize_nvfp4_activation"](a[t:t + 1]) for t in range(a.shape[0])])
    return _orig["quantize_nvfp4_activation"](a)


def _nvfp4_h_unquantised(hs):
    return hs


def _q8_0_x_unquantised_in_layer(a):
    # wiring mistake: Layer.forward skips the Q8_0 step of x (its h step still runs)
    if _called_from_layer_forward():
        return np.asarray(a, np.float64)
    return _orig["quantize_q8_0_activation"](a)


MUTANTS = {
    "decode_int4/nibbles_swapped": ("decode_int4", _nibbles_swapped),
    "decode_int4/unsigned": ("decode_int4", _unsigned_int4),
    "dequant_int4_g32/scale_group_shift": ("dequant_int4_g32", _scale_group_shift),
    "decode_e4m3/bias8": ("decode_e4m3", _e4m3_bias8),
    "decode_e2m1/subnormal": ("decode_e2m1", _e2m1_subnormal),
    "sigmoid/sign": ("sigmoid", _sigmoid_sign),
    "silu/sign": ("silu", _silu_sign),
    "swiglu/gate_up_swapped": ("swiglu_hidden", _swiglu_swapped),
    "down_proj/transposed": ("down_proj", _down_transposed),
    "select/top1_group_score": ("select_experts", _select_top1_group),
    "select/zero_fill": ("select_experts", _select_zero_fill),
    "select/ties_high": ("select_experts", _select_ties_high),
    "select/bias_ignored": ("select_experts", _select_bias_ignored),
    "weights/no_rsf": ("routing_weights", _weights_no_rsf),
    "weights/unnormalised": ("routing_weights", _weights_unnormalised),
    "group/descending": ("group_tokens", _group_descending),
    "nvfp4_act/scale": ("quantize_nvfp4_activation", _act_scale_no6),
    "nvfp4_layer/h_scale_per_expert": ("quantize_routed_h", _h_scale_per_expert),
    "nvfp4_layer/shared_reads_quantised_x": ("shared_expert_input", _shared_reads_quantised_x),
    "widen_bf16/truncating": ("widen_bf16", _widen_bf16_truncating),
    "top_p/boundary_inclusive": ("expert_top_p", lambda s, i, p: _top_p_variant(s, i, p, le=True)),
    "top_p/slot_order": ("expert_top_p", lambda s, i, p: _top_p_variant(s, i, p, slot_order=True)),
    "top_p/ties_high": ("expert_top_p", lambda s, i, p: _top_p_variant(s, i, p, ties_high=True)),
    "weights/dropped_unmasked": ("routing_weights", _weights_dropped_unmasked),
    "group/dropped_counted": ("group_tokens", _group_dropped_counted),
    "int_row/fields_reversed": ("decode_int_row", _int_row_fields_reversed),
    "int_row/unsigned": ("decode_int_row", _int_row_unsigned),
    "q8_0/no_fp16_step": ("quantize_q8_0_activation", _q8_0_no_fp16_step),
    "q8_0/round_half_up": ("quantize_q8_0_activation", _q8_0_round_half_up),
    "q8_0_layer/h_unquantised": ("quantize_q8_0_activation", _q8_0_h_unquantised),
    "select/group_sum_all": ("select_experts", _select_variant("group_sum_all")),
    "select/no_group_mask": ("select_experts", _select_variant("no_group_mask")),
    "select/groups_by_unbiased_scores": ("select_experts", _select_variant("groups_unbiased")),
    "sigmoid/softmax": ("sigmoid", _softmax),
    "weights/slot_rolled": ("routing_weights", _weights_slot_rolled),
    "silu/without_x": ("silu", _silu_without_x),
    "widen_bf16/as_fp16": ("widen_bf16", _widen_as_fp16),
    "decode_e4m3/no_subnormal": ("decode_e4m3", _e4m3_no_subnormal),
    "decode_e2m1/sign_ignored": ("decode_e2m1", _e2m1_sign_ignored),
    "q8_0/block16": ("quantize_q8_0_activation", _q8_0_block16),
    "dequant_int_row/scale_ignored": ("dequant_int_row", _int_row_scale_ignored),
    "group/slot_major": ("group_tokens", _group_slot_major),
    "nvfp4_act/e2m1_ties_away": ("nvfp4_activation_parts", _nvfp4_parts_variant("e2m1_ties_away")),
    "nvfp4_act/e4m3_scale_truncated": ("nvfp4_activation_parts", _nvfp4_parts_variant("e4m3_truncated")),
    "nvfp4_act/tensor_scale_per_row": ("nvfp4_activation_parts", _nvfp4_parts_variant("ts_per_row")),
    "nvfp4_act/block_amax_per_32": ("nvfp4_activation_parts", _nvfp4_parts_variant("amax32")),
    "nvfp4_act/tensor_scale_without_6": ("nvfp4_activation_parts", _nvfp4_parts_variant("ts_no6")),
    "dequant_nvfp4/tensor_scale_ignored": ("dequant_nvfp4", _nvfp4_tensor_scale_ignored),
    "dequant_nvfp4/scale_per_32": ("dequant_nvfp4", _nvfp4_scale_per_32),
    "decode_e4m3/no_nan": ("decode_e4m3", _e4m3_no_nan),
    "dequant_int4_g32/scale_per_16": ("dequant_int4_g32", _int4_scale_per_16),
    "q8_0/divide_by_128": ("quantize_q8_0_activation", _q8_0_divide_by_128),
    "top_p/mass_of_all_experts": ("expert_top_p", _top_p_rule_variant("mass_of_all_E")),
    "top_p/crossing_expert_dropped": ("expert_top_p", _top_p_rule_variant("crossing_dropped")),
    "top_p/ranked_by_id": ("expert_top_p", _top_p_rule_variant("order_by_id")),
    "top_p/margin_zero": ("expert_top_p", _top_p_margin_zero),
    "select/margins_zero": ("select_experts", _select_margins(0.0)),
    "select/margins_inf": ("select_experts", _select_margins(np.inf)),
    "router/fp32": ("router_logits", _router_fp32),
    "sigmoid/fp32": ("sigmoid", _sigmoid_fp32),
    "silu/fp32": ("silu", _silu_fp32),
    "group/token_only": ("group_tokens", _group_token_only),
    "identity_glu/up_only": ("identity_glu_hidden", _identity_glu_up_only),
    "nvfp4_layer/x_unquantised": ("quantize_nvfp4_activation", _nvfp4_x_unquantised_in_layer),
    "nvfp4_layer/x_tensor_scale_per_token": ("quantize_nvfp4_activation", _nvfp4_x_per_token_in_layer),
    "nvfp4_layer/h_unquantised": ("quantize_routed_h", _nvfp4_h_unquantised),
    "q8_0_layer/x_unquantised": ("quantize_q8_0_activation", _q8_0_x_unquantised_in_layer),
}


def _some_pin_fails() -> bool:
    for pin in P.ALL_PINS:
        try:
            pin(O)
        except (AssertionError, ValueError, IndexError):
            return True
    return False


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    assert _some_pin_fails(), f"no pin caught the planted mistake {name}"


def test_shared_weighted_by_rsf_is_caught(monkeypatch):
    orig = O.Layer.shared_expert

    def scaled(self):
        gu, d = orig(self)
        return gu, d * self.rsf

    monkeypatch.setattr(O.Layer, "shared_expert", scaled)
    assert _some_pin_fails()


def test_layer_ignoring_top_p_is_caught(monkeypatch):
    # a wiring mistake of the layer: the selection is used without the adaptive top-p cut
    monkeypatch.setattr(O, "expert_top_p",
                        lambda s, i, p: O.TopP(np.ones(np.shape(i), bool), np.full(np.shape(i)[0], np.inf)))
    assert _some_pin_fails()


def test_layer_weights_from_biased_scores_is_caught(monkeypatch):
    # a wiring mistake of the layer: the combine weights (and the top-p cut) use the biased
    # scores b = s + bias, which noaux_tc uses for the selection only
    orig = O.Layer.route

    def route(self, x64):
        scores, sel = orig(self, x64)
        return scores + np.asarray(self.a["bias"], np.float64)[None], sel

    monkeypatch.setattr(O.Layer, "route", route)
    assert _some_pin_fails()


def test_unmutated_oracle_passes_every_pin():
    assert not _some_pin_fails()
