"""fp64 CPU oracle of the quantised routed-MoE layer forward.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg and ``--impl reference`` arm may import this module; the library's own
path never does, and it shares no code with the CUDA sources.

What it computes, step by step, in the pages' order (DeepSeek-V3-style router with
noaux_tc, routed_scaling_factor and an always-on shared expert: "Show HN: Menjalankan
GLM 5.2 di komputer lambat", section "Fitur utama yang diimplementasikan"; batch-union
MoE: same page and section, and "16 Teknik Özellik ve Yazılım Çıkarımları" on the
Turkish restatement; NVFP4 experts with FP8 scales per 16 elements: "NVIDIA stellt
neues GLM-5.2 NVFP4 Modell vor", section "Technische Details und Quantisierungsansatz"):

1. logits l = x W_r^T (fp64, on the exactly widened x and W_r);
2. gate scores s = sigmoid(l);
3. biased scores b = s + bias; the bias only selects (auxiliary-loss-free balancing);
4. group score = sum of the two largest b of each contiguous group of E/n_group experts;
5. keep the topk_group best groups; experts of other groups are excluded (-inf);
6. ids = the top_k largest b among kept experts; ties go to the lower index, for
   groups and for experts;
7. w = s[ids] / sum(s[ids]) * routed_scaling_factor (unbiased s); with the adaptive
   expert top-p (the "--topp" option of the first page, section "Mengunduh model dan
   menjalankannya") the slots outside the shortest score-ordered prefix reaching p of the
   mass are dropped (id -1, weight 0) and the sum runs over the kept slots;
8. batch-union grouping: per expert, the (token, slot) entries that chose it, in
   ascending token order; entry = token * top_k + slot;
9. per (token, expert): gu = W_gu x_t; h = SiLU(gu[:I]) * gu[I:]; y = W_d h, with the
   weights dequantised exactly (int4 code * fp16 scale, E2M1 code * E4M3 block scale
   * fp32 tensor scale, or an int8 / int4 / int2 code * its row's fp32 scale: the per-row
   formats of "Fitur utama yang diimplementasikan"); with Q8_0-style activations (same
   section) x and every h are rounded to int8 codes with an fp16 step per 32 elements
   before their matmul;
10. out_t = sum_j w[t, j] y_{t, ids[t, j]} + y_{t, shared}; the shared expert has weight 1.

NVFP4 layers also quantise the activations that feed the routed experts (x before the
gate/up projection, h before the down projection) to NVFP4 with a per-call tensor scale
(one scale over all tokens of x; one over all routed h rows of the call); the router and a
bf16 shared expert read the unquantised x. The codes are decided in fp32: the format's
tensor scale is an fp32 number by definition, and the block scale and each element's code
are the E4M3 and E2M1 roundings of quotients by it, so those quotients are fp32
operations (an fp64 quotient could fall on the other side of a rounding boundary); the
dequantised values are then used exactly.

Readings where the pages are silent are stated at each function. Every function here is
pinned by ``tests/test_oracle_pins.py`` to something other than itself (brute force,
closed forms, hand-worked fixtures, format definitions, library routines).
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# ------------------------------------------------------------------ storage decoders


def _int4_pair_table() -> np.ndarray:
    """[256, 2] int64: the (low, high) two's-complement nibble values of every byte."""
    b = np.arange(256)
    lo, hi = b & 0x0F, b >> 4
    return np.stack([np.where(lo >= 8, lo - 16, lo), np.where(hi >= 8, hi - 16, hi)], axis=1)


_INT4_PAIRS = _int4_pair_table()


def decode_int4(codes: np.ndarray) -> np.ndarray:
    """Packed two's-complement int4 -> int64, element 2j from the low nibble of byte j,
    2j+1 from the high nibble (the packed int4 container of "Fitur utama yang
    diimplementasikan")."""
    codes = np.asarray(codes, dtype=np.uint8)
    return _INT4_PAIRS[codes].reshape(*codes.shape[:-1], codes.shape[-1] * 2)


_INT4_LO = _INT4_PAIRS[:, 0].astype(np.float64)
_INT4_HI = _INT4_PAIRS[:, 1].astype(np.float64)


def dequant_int4_g32(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """W[n, k] = code[n, k] * scale[n, k // 32], exact in fp64 (dequant-on-use of the
    packed int4 weights; one fp16 scale per 32 input-dim elements)."""
    codes = np.asarray(codes, dtype=np.uint8)
    n, kb = codes.shape
    k = 2 * kb
    c = np.empty((n, k))
    np.take(_INT4_LO, codes, out=c[:, 0::2])
    np.take(_INT4_HI, codes, out=c[:, 1::2])
    s = np.asarray(scales, dtype=np.float16).astype(np.float64)
    assert s.shape == (n, k // 32)
    c = c.reshape(n, k // 32, 32)
    c *= s[..., None]
    return c.reshape(n, k)


def decode_e2m1(nibbles: np.ndarray) -> np.ndarray:
    """FP4 E2M1 (1 sign, 2 exponent bits with bias 1, 1 mantissa bit; exponent field 0
    is subnormal with step 0.5) -> fp64."""
    n = np.asarray(nibbles, dtype=np.int64) & 0xF
    sign = np.where(n & 8, -1.0, 1.0)
    e = (n >> 1) & 3
    m = n & 1
    mag = np.where(e == 0, 0.5 * m, (1.0 + 0.5 * m) * np.exp2(e - 1.0))
    return sign * mag


def decode_e4m3(bits: np.ndarray) -> np.ndarray:
    """FP8 E4M3 (bias 7, subnormal step 2^-9, no infinities, S.1111.111 is NaN) -> fp64."""
    b = np.asarray(bits, dtype=np.int64) & 0xFF
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((b & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


_E2M1_LO = decode_e2m1(np.arange(256) & 0x0F)   # value of the low nibble of every byte
_E2M1_HI = decode_e2m1(np.arange(256) >> 4)     # and of the high nibble
_E4M3_ALL = decode_e4m3(np.arange(256))          # value of every E4M3 byte


def dequant_nvfp4(codes: np.ndarray, scales: np.ndarray, tensor_scale) -> np.ndarray:
    """W[n, k] = e2m1(code[n, k]) * e4m3(scale[n, k // 16]) * tensor_scale, exact in fp64
    (NVFP4: 4-bit elements, an FP8 scale per 16 elements, one fp32 scale per tensor).
    Element 2j is the low nibble of byte j; the byte tables are the decoders above applied
    to every byte value."""
    codes = np.asarray(codes, dtype=np.uint8)
    n, kb = codes.shape
    k = 2 * kb
    c = np.empty((n, k))
    np.take(_E2M1_LO, codes, out=c[:, 0::2])
    np.take(_E2M1_HI, codes, out=c[:, 1::2])
    sb = _E4M3_ALL[np.asarray(scales, dtype=np.uint8)]
    assert sb.shape == (n, k // 16)
    c = c.reshape(n, k // 16, 16)
    c *= sb[..., None]
    c = c.reshape(n, k)
    c *= float(np.float32(tensor_scale))
    return c


def decode_int_row(codes: np.ndarray, bits: int) -> np.ndarray:
    """Packed two's-complement integers of the per-row formats -> int64 [N, K]: int8 one
    per byte; int4 two per byte (element 2j in the low nibble of byte j); int2 four per byte
    (element 4j + i in bits 2i..2i+1 of byte j)."""
    c = np.asarray(codes, np.uint8).astype(np.int64)
    per = 8 // bits
    fields = np.stack([(c >> (bits * i)) & ((1 << bits) - 1) for i in range(per)], axis=-1)
    v = fields.reshape(c.shape[:-1] + (c.shape[-1] * per,))
    return np.where(v >= 1 << (bits - 1), v - (1 << bits), v)


def dequant_int_row(codes: np.ndarray, scales: np.ndarray, bits: int) -> np.ndarray:
    """Per-row symmetric integer weights (the "int8, packed int4, packed int2, scale per-row"
    formats of "Show HN: Menjalankan GLM 5.2 di komputer lambat", section "Fitur utama yang
    diimplementasikan"): w[n, k] = code[n, k] * scale[n], one fp32 scale per row."""
    return decode_int_row(codes, bits) * np.asarray(scales, np.float64).reshape(-1, 1)


def quantize_q8_0_activation(a: np.ndarray) -> np.ndarray:
    """Q8_0-style int8 activations (the integer-dot kernels' activations of "Show HN:
    Menjalankan GLM 5.2 di komputer lambat", section "Fitur utama yang diimplementasikan").
    The pages name the style only; reading: per 32 consecutive elements of a row, d =
    fp16_rne(amax / 127) and q = clamp(rint_even(a / d), -127, 127) (d = 0 gives q = 0),
    both quotients fp32 operations on the fp32 value of a; returns q * d (fp64)."""
    a32 = np.asarray(a, np.float32)
    m, k = a32.shape
    blocks = a32.reshape(m, k // 32, 32)
    amax = np.max(np.abs(blocks), axis=2)
    d = (amax / np.float32(127.0)).astype(np.float32).astype(np.float16).astype(np.float32)
    q = np.zeros(blocks.shape, np.float32)
    np.divide(blocks, d[..., None], out=q, where=d[..., None] != 0)
    q = np.clip(np.rint(q), -127, 127)
    return (q.astype(np.float64) * d[..., None].astype(np.float64)).reshape(m, k)


ROW_FORMAT_BITS = {"int8_row": 8, "int4_row": 4, "int2_row": 2}


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp64 (exact)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


# ----------------------------------------------------- NVFP4 activation quantiser


_E2M1_MAGS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e4m3_mags() -> np.ndarray:
    return np.array([decode_e4m3(np.array([c]))[0] for c in range(0x7F)])


_E4M3_MAGS = _e4m3_mags()


def _rne_code(mag: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Index into ``table`` (ascending magnitudes, index parity = mantissa parity) of the
    value nearest to ``mag``; halfway cases take the even index; saturates at the top."""
    mag = np.asarray(mag, dtype=np.float64)
    j = np.clip(np.searchsorted(table, mag, side="right") - 1, 0, len(table) - 2)
    below = mag - table[j]          # table[j] <= mag < table[j + 1] inside the range
    above = table[j + 1] - mag
    up = (above < below) | ((above == below) & (j % 2 == 1))
    return np.where(mag >= table[-1], len(table) - 1, j + up).astype(np.int64)


def nvfp4_activation_parts(a: np.ndarray):
    """NVFP4 quantisation of a [M, K] activation, as its three parts: the E2M1 element
    values [M, K/16, 16] (signed, fp64), the E4M3 block scales [M, K/16] (fp64) and the fp32
    tensor scale.

    Reading of the NVFP4 scheme for activations (the pages give only "FP8 scales per 16
    elements"): one dynamic fp32 tensor scale per call, ts = amax(|a|) / (6 * 448); per
    16-element block, scale = E4M3_rne_satfinite((amax16 / 6) / ts); element code =
    E2M1_rne_satfinite(a / (scale * ts)). Every quotient and product that decides a code
    is an fp32 operation, in this order, on the fp32 value of ``a``. ts = 0 gives zero
    scales and codes.
    """
    a32 = np.asarray(a, dtype=np.float32)
    m, k = a32.shape
    amax = np.float32(np.max(np.abs(a32))) if a32.size else np.float32(0)
    ts = np.float32(amax / np.float32(2688.0))
    if ts == 0:
        return np.zeros((m, k // 16, 16)), np.zeros((m, k // 16)), ts
    blocks = a32.reshape(m, k // 16, 16)
    bamax = np.max(np.abs(blocks), axis=2)
    ratio = ((bamax / np.float32(6.0)).astype(np.float32) / ts).astype(np.float32)
    sb = _E4M3_MAGS[_rne_code(ratio, _E4M3_MAGS)]
    denom = (sb.astype(np.float32) * ts).astype(np.float32)
    q = np.zeros(blocks.shape, np.float32)
    np.divide(blocks, denom[..., None], out=q, where=denom[..., None] != 0)
    mag = _E2M1_MAGS[_rne_code(np.abs(q), _E2M1_MAGS)]
    return np.sign(q) * mag, sb, ts


def quantize_nvfp4_activation(a: np.ndarray) -> np.ndarray:
    """Quantise a [M, K] activation to NVFP4 (nvfp4_activation_parts) and return the
    dequantised values code * block scale * tensor scale (fp64)."""
    m, k = np.shape(a)
    code_val, sb, ts = nvfp4_activation_parts(a)
    return (code_val * sb[..., None] * float(ts)).reshape(m, k)


# ----------------------------------------------------------------------- router


def router_logits(x: np.ndarray, router_w: np.ndarray) -> np.ndarray:
    """l[t, e] = sum_h x[t, h] W_r[e, h] in fp64 (the router projection)."""
    return np.asarray(x, np.float64) @ np.asarray(router_w, np.float64).T


def sigmoid(z: np.ndarray) -> np.ndarray:
    """Gate score of the sigmoid router: 1 / (1 + e^-z)."""
    return 1.0 / (1.0 + np.exp(-z))


@dataclass
class Selection:
    ids: np.ndarray          # [T, top_k] int64, slot order = descending b, ties lower id
    group_margin: np.ndarray  # [T] gap between the last kept and the first dropped group
    expert_margin: np.ndarray  # [T] gap between the k-th and (k+1)-th kept expert

    @property
    def margin(self) -> np.ndarray:
        return np.minimum(self.group_margin, self.expert_margin)


def select_experts(scores: np.ndarray, bias: np.ndarray, n_group: int, topk_group: int,
                   top_k: int) -> Selection:
    """noaux_tc grouped top-k on the biased scores b = s + bias.

    Group score = sum of the two largest b in each contiguous group; the topk_group
    best groups are kept; the top_k largest b among kept experts are selected. Ties go
    to the lower index at both levels (stable descending order). Experts outside kept
    groups are excluded outright (-inf), not zeroed.
    """
    s = np.asarray(scores, np.float64)
    t_count, n_exp = s.shape
    g_size = n_exp // n_group
    if g_size * n_group != n_exp or g_size < 2 or not 1 <= topk_group <= n_group \
            or not 1 <= top_k <= topk_group * g_size:
        raise ValueError("invalid routing shape")
    b = s + np.asarray(bias, np.float64)[None, :]
    ids = np.empty((t_count, top_k), np.int64)
    gm = np.full(t_count, np.inf)
    em = np.full(t_count, np.inf)
    for t in range(t_count):
        grp = b[t].reshape(n_group, g_size)
        top2 = -np.sort(-grp, axis=1)[:, :2]
        gscore = top2[:, 0] + top2[:, 1]
        g_order = np.argsort(-gscore, kind="stable")
        kept = g_order[:topk_group]
        if topk_group < n_group:
            gm[t] = gscore[g_order[topk_group - 1]] - gscore[g_order[topk_group]]
        masked = np.full(n_exp, -np.inf)
        for g in kept:
            masked[g * g_size:(g + 1) * g_size] = b[t, g * g_size:(g + 1) * g_size]
        e_order = np.argsort(-masked, kind="stable")
        ids[t] = e_order[:top_k]
        if top_k < topk_group * g_size:
            em[t] = masked[e_order[top_k - 1]] - masked[e_order[top_k]]
    return Selection(ids, gm, em)


def routing_weights(scores: np.ndarray, ids: np.ndarray, rsf: float) -> np.ndarray:
    """w[t, j] = s[t, ids[t, j]] / sum_j s[t, ids[t, j]] * routed_scaling_factor, the sum
    over the routed slots; a slot dropped by the adaptive top-p (id -1) has weight 0."""
    ids = np.asarray(ids)
    routed = ids >= 0
    sel = np.where(routed, np.take_along_axis(np.asarray(scores, np.float64), np.where(routed, ids, 0), axis=1),
                   0.0)
    return sel / sel.sum(axis=1, keepdims=True) * float(np.float32(rsf))


def group_tokens(ids: np.ndarray, n_experts: int):
    """Batch-union grouping: counts[E], offsets[E+1] (exclusive scan) and the entry list
    holding token*top_k + slot of every routed slot (id >= 0), grouped by expert, ascending
    token in each group."""
    t_count, k = ids.shape
    flat = np.asarray(ids).ravel()
    counts = np.bincount(flat[flat >= 0], minlength=n_experts)[:n_experts]
    offsets = np.zeros(n_experts + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    lst = np.empty(int(offsets[-1]), np.int64)
    cursor = offsets[:-1].copy()
    for t in range(t_count):
        for j in range(k):
            e = ids[t, j]
            if e < 0:
                continue
            lst[cursor[e]] = t * k + j
            cursor[e] += 1
    return counts, offsets, lst


# ------------------------------------------------------- adaptive expert top-p


@dataclass
class TopP:
    keep: np.ndarray     # [T, top_k] bool: the slot stays routed
    margin: np.ndarray   # [T] distance of the decision from its threshold (relative), inf if none


def expert_top_p(scores: np.ndarray, ids: np.ndarray, p: float) -> TopP:
    """Adaptive expert top-p (the "--topp" option of "Show HN: Menjalankan GLM 5.2 di komputer
    lambat", section "Mengunduh model dan menjalankannya": fewer experts per token, less
    expert data read; section "Benchmark komunitas" for its effect). The pages do not state
    the rule. Reading: order the top_k experts the selection chose by their unbiased score s,
    largest first (equal scores: lower expert index first), and keep the shortest prefix
    whose summed s reaches p times the summed s of all top_k: an expert stays when the mass
    ranked before it is below p times the total, so the first always stays. p <= 0 or p >= 1
    keeps every slot. margin[t]: the smallest |mass before rank r - p * total| over r >= 1,
    and the score gap across the cut, each divided by the total."""
    s = np.asarray(scores, np.float64)
    ids = np.asarray(ids, np.int64)
    t_count, k = ids.shape
    keep = np.ones((t_count, k), bool)
    margin = np.full(t_count, np.inf)
    if not 0.0 < p < 1.0:
        return TopP(keep, margin)
    for t in range(t_count):
        sel = s[t, ids[t]]
        order = np.lexsort((ids[t], -sel))          # s descending, then lower id
        ranked = sel[order]
        total = ranked.sum()
        before = np.concatenate([[0.0], np.cumsum(ranked)[:-1]])
        kept = before < p * total
        keep[t, order] = kept
        if k > 1:
            m = np.min(np.abs(before[1:] - p * total))
            n_kept = int(kept.sum())
            if n_kept < k:
                m = min(m, ranked[n_kept - 1] - ranked[n_kept])
            margin[t] = m / total
    return TopP(keep, margin)


# ------------------------------------------------------------------- expert FFN


def silu(z: np.ndarray) -> np.ndarray:
    """SiLU(z) = z * sigmoid(z)."""
    return z / (1.0 + np.exp(-z))


def swiglu_hidden(w_gu: np.ndarray, xr: np.ndarray) -> np.ndarray:
    """h = SiLU(gate) * up with [gate; up] = W_gu x (rows 0..I-1 gate, I..2I-1 up)."""
    gu = np.asarray(xr, np.float64) @ np.asarray(w_gu, np.float64).T
    i = gu.shape[1] // 2
    return silu(gu[:, :i]) * gu[:, i:]


def identity_glu_hidden(w_gu: np.ndarray, xr: np.ndarray) -> np.ndarray:
    """h = gate * up, the gated unit with the SiLU bypassed. Test-only: with integer
    activations and power-of-two scales every step of the layer is then exact in fp64 and
    in fp32, so an implementation's expert and combine arithmetic can be compared bit for
    bit (the layer itself always uses SiLU)."""
    gu = np.asarray(xr, np.float64) @ np.asarray(w_gu, np.float64).T
    i = gu.shape[1] // 2
    return gu[:, :i] * gu[:, i:]


def down_proj(w_d: np.ndarray, h: np.ndarray) -> np.ndarray:
    """y = W_d h."""
    return np.asarray(h, np.float64) @ np.asarray(w_d, np.float64).T


# ---------------------------------------------------- NVFP4 layer activation rules


def quantize_routed_h(hs: dict) -> dict:
    """NVFP4 h before the routed experts' down projections (reading of the NVFP4 layer:
    one per-call tensor scale covers every routed h row of the call, like x's covers every
    token). ``hs`` maps expert -> (entries, h rows); the rows of all experts, in ascending
    expert order, form one activation for quantize_nvfp4_activation."""
    order = sorted(hs)
    h_q = quantize_nvfp4_activation(np.concatenate([hs[e][1] for e in order]).astype(np.float32))
    out, n0 = {}, 0
    for e in order:
        n1 = n0 + len(hs[e][0])
        out[e] = (hs[e][0], h_q[n0:n1])
        n0 = n1
    return out


def shared_expert_input(shared_format: str, x64: np.ndarray, x_in: np.ndarray) -> np.ndarray:
    """Activation the shared expert reads: a bf16 shared expert (the NVFP4 layer keeps it
    unquantised, like the router) reads the unquantised x; a shared expert stored in the
    routed format reads the same activation as the routed experts."""
    return x64 if shared_format == "bf16" else x_in


# ----------------------------------------------------------------- whole layer


@dataclass
class LayerRef:
    """Oracle outputs of one forward."""

    out: np.ndarray            # [T, H] fp64
    ids: np.ndarray            # [T, k]
    weights: np.ndarray        # [T, k]
    scores: np.ndarray         # [T, E] unbiased sigmoid scores
    margin: np.ndarray         # [T]
    counts: np.ndarray
    offsets: np.ndarray
    entries: np.ndarray


class Layer:
    """Weights of one layer as the oracle sees them (dequantised lazily, per expert)."""

    def __init__(self, arrays: dict, *, hidden, inter, n_experts, top_k, n_group, topk_group,
                 rsf, weight_format, act_dtype, router_dtype, shared_format, expert_top_p=0.0,
                 act_quant="none"):
        self.a = arrays
        self.H, self.I, self.E = hidden, inter, n_experts
        self.top_k, self.n_group, self.topk_group = top_k, n_group, topk_group
        self.rsf = rsf
        self.expert_top_p = expert_top_p
        if act_quant not in ("none", "q8_0") or (act_quant == "q8_0" and shared_format != weight_format):
            raise ValueError(act_quant)
        self.act_quant = act_quant
        self.weight_format, self.act_dtype = weight_format, act_dtype
        self.router_dtype, self.shared_format = router_dtype, shared_format

    @classmethod
    def from_spec(cls, spec, arrays: dict) -> "Layer":
        return cls(arrays, hidden=spec.hidden, inter=spec.inter, n_experts=spec.n_experts,
                   top_k=spec.top_k, n_group=spec.n_group, topk_group=spec.topk_group,
                   rsf=spec.rsf, weight_format=spec.weight_format, act_dtype=spec.act_dtype,
                   router_dtype=spec.router_dtype, shared_format=spec.shared_format,
                   expert_top_p=getattr(spec, "expert_top_p", 0.0),
                   act_quant=getattr(spec, "act_quant", "none"))

    # -- weights
    def router_w(self) -> np.ndarray:
        w = self.a["router_w"]
        return widen_bf16(w) if self.router_dtype == "bf16" else np.asarray(w, np.float64)

    def _matrix(self, prefix: str, idx: int, fmt: str, which: str) -> np.ndarray:
        """One dequantised expert matrix: which = "gu" (W_gu [2I, H]) or "d" (W_d [H, I])."""
        a, p = self.a, prefix + which
        if fmt == "int4_g32":
            return dequant_int4_g32(a[p + "_codes"][idx], a[p + "_scales"][idx])
        if fmt == "nvfp4":
            return dequant_nvfp4(a[p + "_codes"][idx], a[p + "_scales"][idx], a[p + "_tscale"][idx])
        if fmt == "bf16":
            return widen_bf16(a[p + "_bf16"][idx])
        if fmt in ROW_FORMAT_BITS:
            return dequant_int_row(a[p + "_codes"][idx], a[p + "_scales"][idx], ROW_FORMAT_BITS[fmt])
        raise ValueError(fmt)

    def routed_gu(self, e: int) -> np.ndarray:
        return self._matrix("", e, self.weight_format, "gu")

    def routed_d(self, e: int) -> np.ndarray:
        return self._matrix("", e, self.weight_format, "d")

    def routed_expert(self, e: int):
        return self.routed_gu(e), self.routed_d(e)

    def shared_expert(self):
        return (self._matrix("sh_", 0, self.shared_format, "gu"),
                self._matrix("sh_", 0, self.shared_format, "d"))

    def widen_x(self, x: np.ndarray) -> np.ndarray:
        return widen_bf16(x) if self.act_dtype == "bf16" else np.asarray(x, np.float64)

    # -- forward
    def route(self, x64: np.ndarray):
        scores = sigmoid(router_logits(x64, self.router_w()))
        sel = select_experts(scores, self.a["bias"], self.n_group, self.topk_group, self.top_k)
        return scores, sel

    def forward(self, x: np.ndarray, ids: np.ndarray | None = None,
                tokens: np.ndarray | None = None, activation: str = "silu") -> LayerRef:
        """Whole-layer forward. ``ids`` overrides the selection (used to re-run the
        oracle on a near-tie token with the selection another implementation made);
        ``tokens`` restricts the expert FFNs and the output to those rows (the routing
        and the NVFP4 activation scales still see every token); ``activation`` =
        "identity" bypasses the SiLU (test-only exact-arithmetic cases)."""
        if activation not in ("silu", "identity"):
            raise ValueError(activation)
        hidden = swiglu_hidden if activation == "silu" else identity_glu_hidden
        x64 = self.widen_x(x)
        t_count = x64.shape[0]
        scores, sel = self.route(x64)
        margin = sel.margin
        if ids is None:
            # adaptive expert top-p: dropped slots get id -1 (no-op unless 0 < p < 1)
            tp = expert_top_p(scores, sel.ids, self.expert_top_p)
            use_ids = np.where(tp.keep, sel.ids, -1)
            margin = np.minimum(margin, tp.margin)
        else:
            use_ids = np.asarray(ids, np.int64)
        w = routing_weights(scores, use_ids, self.rsf)
        counts, offsets, entries = group_tokens(use_ids, self.E)
        rows = np.arange(t_count) if tokens is None else np.asarray(tokens, np.int64)
        want = np.zeros(t_count, bool)
        want[rows] = True
        out = np.zeros((t_count, self.H))

        nvfp4 = self.weight_format == "nvfp4"
        q8 = self.act_quant == "q8_0"
        x_in = quantize_nvfp4_activation(x64.astype(np.float32)) if nvfp4 else x64
        if q8:      # int8 activations into every expert matmul (x here, h below)
            x_in = quantize_q8_0_activation(x64)
            hidden_in = hidden

            def hidden(w_gu, xr):
                return quantize_q8_0_activation(hidden_in(w_gu, xr))

        # routed experts, batch-union: each expert's weights applied to all its tokens
        hs = {}      # e -> (entries, h rows)
        for e in range(self.E):
            ent = entries[offsets[e]:offsets[e + 1]]
            if not nvfp4:    # an NVFP4 layer needs every routed h for the h tensor scale
                ent = ent[want[ent // self.top_k]]
            if ent.size == 0:
                continue
            hs[e] = (ent, hidden(self.routed_gu(e), x_in[ent // self.top_k]))
        if nvfp4 and hs:
            hs = quantize_routed_h(hs)
        for e, (ent, h) in hs.items():
            keep = want[ent // self.top_k]
            if not keep.any():
                continue
            y = down_proj(self.routed_d(e), h[keep])
            for r, yy in zip(ent[keep], y):
                t, j = divmod(int(r), self.top_k)
                out[t] += w[t, j] * yy

        sh_gu, sh_d = self.shared_expert()
        xs = shared_expert_input(self.shared_format, x64, x_in)[rows]
        out[rows] += down_proj(sh_d, hidden(sh_gu, xs))
        return LayerRef(out, use_ids, w, scores, margin, counts, offsets, entries)
