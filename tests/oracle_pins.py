"""Pins of the fp64 oracle: each check ties an oracle function to something other than
itself (a format definition, a library routine, brute force, a closed form, an
invariant). Every pin reads the oracle through the module object it is given, so the
mutation tests can hand it a deliberately broken oracle and watch a pin fail.
"""

from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------------------ helpers


def pack_int4_rows(codes: np.ndarray) -> np.ndarray:
    """Pack int codes in [-8, 7] row-wise, element 2j in the low nibble of byte j."""
    c = np.asarray(codes, np.int64)
    u = (c & 0xF).astype(np.uint8)
    return (u[..., 0::2] | (u[..., 1::2] << 4)).astype(np.uint8)


def sigmoid_scalar(z: float) -> float:
    return 1.0 / (1.0 + math.exp(-z))


def silu_scalar(z: float) -> float:
    return z * sigmoid_scalar(z)


def hand_layer(O, case: str):
    """Build the hand-worked two-expert layer of tests/golden/hand_two_expert.json."""
    with open(os.path.join(GOLDEN, "hand_two_expert.json")) as f:
        g = json.load(f)
    H, I, E = g["hidden"], g["inter"], g["n_experts"]
    x = np.zeros((1, H), np.float32)
    for k, v in g["x_nonzero"].items():
        x[0, int(k)] = v
    wr = np.zeros((E, H), np.float32)
    for e, row in g["router_w"].items():
        for h, v in row.items():
            wr[int(e), int(h)] = v

    def expert(spec):
        gu = np.zeros((2 * I, H), np.int64)
        gus = np.zeros((2 * I, H // 32), np.float16)
        for r, d in spec["gu"].items():
            gu[int(r), :4] = d["codes"]
            gus[int(r), 0] = d["scale"]
        dd = np.zeros((H, I), np.int64)
        ds = np.zeros((H, I // 32), np.float16)
        for r, d in spec["d"].items():
            dd[int(r), 0] = d["code0"]
            ds[int(r), 0] = d["scale"]
        return pack_int4_rows(gu), gus, pack_int4_rows(dd), ds

    ex = [expert(s) for s in g["experts"]]
    sh = expert(g["shared"])
    c = g["cases"][case]
    arrays = {
        "router_w": wr, "bias": np.array(c["bias"], np.float32),
        "gu_codes": np.stack([e[0] for e in ex]), "gu_scales": np.stack([e[1] for e in ex]),
        "d_codes": np.stack([e[2] for e in ex]), "d_scales": np.stack([e[3] for e in ex]),
        "sh_gu_codes": sh[0][None], "sh_gu_scales": sh[1][None],
        "sh_d_codes": sh[2][None], "sh_d_scales": sh[3][None],
    }
    layer = O.Layer(arrays, hidden=H, inter=I, n_experts=E, top_k=c["top_k"], n_group=1,
                    topk_group=1, rsf=g["rsf"], weight_format="int4_g32", act_dtype="f32",
                    router_dtype="f32", shared_format="int4_g32")
    return layer, x


_E2M1_CODE = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}


def _bf16_bits(v: float) -> int:
    """bf16 bit pattern of a value that bf16 holds exactly (the top half of its fp32 bits)."""
    b = int(np.array([v], np.float32).view(np.uint32)[0])
    assert b & 0xFFFF == 0, v
    return b >> 16


def hand_nvfp4_layer(O):
    """Build the hand-worked NVFP4 layer of tests/golden/hand_nvfp4_layer.json."""
    with open(os.path.join(GOLDEN, "hand_nvfp4_layer.json")) as f:
        g = json.load(f)
    H, I, E = g["hidden"], g["inter"], g["n_experts"]
    x = np.zeros((1, H), np.uint16)
    for k, v in g["x_nonzero"].items():
        x[0, int(k)] = _bf16_bits(v)
    wr = np.zeros((E, H), np.uint16)
    for e, row in g["router_w"].items():
        for h, v in row.items():
            wr[int(e), int(h)] = _bf16_bits(v)

    def nvfp4(rows, K, spec):
        nib = np.zeros((rows, K), np.uint8)
        for r, cols in spec.items():
            for c, v in cols.items():
                nib[int(r), int(c)] = _E2M1_CODE[abs(v)] | (8 if v < 0 else 0)
        packed = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
        return packed, np.full((rows, K // 16), 0x38, np.uint8), np.float32(1.0)

    def bf16(rows, K, spec):
        w = np.zeros((rows, K), np.uint16)
        for r, cols in spec.items():
            for c, v in cols.items():
                w[int(r), int(c)] = _bf16_bits(v)
        return w

    ex = [(nvfp4(2 * I, H, s["gu"]), nvfp4(H, I, s["d"])) for s in g["experts"]]
    arrays = {
        "router_w": wr, "bias": np.zeros(E, np.float32),
        "gu_codes": np.stack([e[0][0] for e in ex]), "gu_scales": np.stack([e[0][1] for e in ex]),
        "gu_tscale": np.array([e[0][2] for e in ex], np.float32),
        "d_codes": np.stack([e[1][0] for e in ex]), "d_scales": np.stack([e[1][1] for e in ex]),
        "d_tscale": np.array([e[1][2] for e in ex], np.float32),
        "sh_gu_bf16": bf16(2 * I, H, g["shared"]["gu"])[None], "sh_d_bf16": bf16(H, I, g["shared"]["d"])[None],
    }
    layer = O.Layer(arrays, hidden=H, inter=I, n_experts=E, top_k=g["top_k"], n_group=1, topk_group=1,
                    rsf=g["rsf"], weight_format="nvfp4", act_dtype="bf16", router_dtype="bf16",
                    shared_format="bf16")
    return layer, x


def brute_force_select(b: np.ndarray, n_group: int, topk_group: int, top_k: int):
    """Exhaustive noaux_tc selection for one token with distinct scores: the best group
    subset by summed group score, then the best expert subset by summed score."""
    E = b.size
    G = E // n_group
    gscore = []
    for g in range(n_group):
        vals = b[g * G:(g + 1) * G]
        best2 = max(vals[i] + vals[j] for i, j in itertools.combinations(range(G), 2))
        gscore.append(best2)
    best_groups = max(itertools.combinations(range(n_group), topk_group),
                      key=lambda gs: sum(gscore[g] for g in gs))
    cand = [e for g in best_groups for e in range(g * G, (g + 1) * G)]
    best = max(itertools.combinations(cand, top_k), key=lambda es: sum(b[e] for e in es))
    return sorted(best)


# --------------------------------------------------------------- storage decoders


def pin_decode_int4(O):
    # two's complement by the machine: shift the nibble to the top of an int8
    b = np.arange(256, dtype=np.uint8)
    lo = (b << 4).astype(np.uint8).view(np.int8) >> 4
    hi = b.view(np.int8) >> 4
    got = O.decode_int4(b[:, None])
    assert np.array_equal(got[:, 0], lo.astype(np.int64))
    assert np.array_equal(got[:, 1], hi.astype(np.int64))
    # hand examples: 0x8F -> (-1, -8), 0x7A -> (-6, 7), 0x21 -> (1, 2)
    assert O.decode_int4(np.array([[0x8F, 0x7A, 0x21]], np.uint8)).tolist() == [[-1, -8, -6, 7, 1, 2]]


def pin_decode_e4m3(O):
    # library routine: torch's float8_e4m3fn for every bit pattern
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.decode_e4m3(np.arange(256))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    # format facts: 0x7E = 448 (largest finite), 0x08 = 2^-6, 0x01 = 2^-9, 0x38 = 1
    assert got[0x7E] == 448.0 and got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def pin_decode_e2m1(O):
    # OCP MX FP4 E2M1 value set, by the sign/exponent/mantissa fields written out
    expected = []
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        mag = (m / 2.0) * 2.0 ** (1 - 1) if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
        expected.append(-mag if s else mag)
    assert np.array_equal(O.decode_e2m1(np.arange(16)), np.array(expected))
    assert list(O.decode_e2m1(np.arange(8))) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def pin_dequant_int4_g32(O):
    codes = np.zeros((2, 64), np.int64)
    codes[0, 0], codes[0, 31], codes[0, 32], codes[1, 63] = 3, -8, 7, -1
    scales = np.array([[0.5, 2.0], [1.0, 0.125]], np.float16)
    w = O.dequant_int4_g32(pack_int4_rows(codes), scales)
    expect = np.zeros((2, 64))
    expect[0, 0], expect[0, 31], expect[0, 32], expect[1, 63] = 1.5, -4.0, 14.0, -0.125
    assert np.array_equal(w, expect)


def pin_dequant_nvfp4(O):
    codes = np.zeros((1, 32), np.int64)
    codes[0, 0], codes[0, 15], codes[0, 16], codes[0, 31] = 0x7, 0xF, 0x3, 0x9   # 6, -6, 1.5, -0.5
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    scales = np.array([[0x38, 0x40]], np.uint8)   # e4m3: 1.0 and 2.0
    w = O.dequant_nvfp4(packed, scales, np.float32(0.25))
    expect = np.zeros((1, 32))
    expect[0, 0], expect[0, 15], expect[0, 16], expect[0, 31] = 1.5, -1.5, 0.75, -0.25
    assert np.array_equal(w, expect)


# ------------------------------------------------------------ activation quantiser


def _brute_round(v: float, table) -> int:
    d = [abs(v - t) for t in table]
    best = min(d)
    cands = [i for i, x in enumerate(d) if x == best]
    even = [i for i in cands if i % 2 == 0]
    return (even or cands)[0]


def pin_nvfp4_rounding(O):
    rng = np.random.default_rng(7)
    # E4M3 rounding against torch's conversion (RNE) on in-range values and exact ties
    grid = O.decode_e4m3(np.arange(0x7F))
    mids = (grid[:-1] + grid[1:]) / 2
    vals = np.concatenate([rng.uniform(0, 440, 2000), rng.uniform(0, 0.02, 2000), mids, grid])
    vals = vals.astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O._rne_code(vals, O._E4M3_MAGS)
    assert np.array_equal(got, ref.astype(np.int64))
    # E2M1 rounding against brute-force nearest-even over the 8 magnitudes
    table = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    vals = np.concatenate([rng.uniform(0, 7, 500), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 9.0]])
    got = O._rne_code(vals, O._E2M1_MAGS)
    want = [7 if v >= 6 else _brute_round(v, table) for v in vals]
    assert got.tolist() == want
    # every representable E2M1 magnitude comes back to its own code, and every code decodes
    # to the magnitude with its sign
    assert O._rne_code(np.array(table, np.float64), O._E2M1_MAGS).tolist() == list(range(8))
    assert O.decode_e2m1(np.arange(8)).tolist() == table
    assert O.decode_e2m1(np.arange(8, 16)).tolist() == [-v for v in table]


def pin_nvfp4_activation(O):
    rng = np.random.default_rng(3)
    # exactly representable input comes back unchanged: with amax 12 the block scales
    # come out as 224, 448 and 112 (exact E4M3 values) and every element sits on the
    # E2M1 grid times its block unit
    a = np.zeros((2, 32), np.float32)
    a[0, :16] = [6, -3, 1.5, 0.5, 0, 4, -2, 1, 6, 0, 0, 0, 0, 0, 0, 0]
    a[0, 16:] = [12, 8, -6, 3, 1, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0]   # block scale 2
    a[1, :16] = [3, 1.5, 0.5, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0]  # block scale 0.5
    deq = O.quantize_nvfp4_activation(a)
    assert np.allclose(deq, a, rtol=1e-6, atol=0), (deq, a)
    # exact ties of the element rounding: with amax 6 the block scale is 448 and the fp32
    # product scale * tensor scale is exactly 1, so each element's quotient is the element
    # itself; 0.25, 1.25, 2.5 and 5.0 lie halfway between E2M1 neighbours and round to the
    # even one (0, 1, 2, 4; signs kept), as round-to-nearest-even does
    a = np.zeros((1, 16), np.float32)
    a[0, :9] = [6.0, 0.25, 1.25, 2.5, 5.0, -0.25, -1.25, -2.5, -5.0]
    vals, sb, ts = O.nvfp4_activation_parts(a)
    assert sb[0, 0] == 448.0 and np.float32(np.float32(sb[0, 0]) * ts) == np.float32(1.0)
    assert vals[0, 0, :9].tolist() == [6.0, 0.0, 1.0, 2.0, 4.0, 0.0, -1.0, -2.0, -4.0], vals[0, 0]
    # error bound on random data: half an E2M1 step at the code's magnitude, relative
    # to the block's scale; at most a quarter of the block scale near zero
    x = rng.standard_normal((8, 64)).astype(np.float32)
    deq = O.quantize_nvfp4_activation(x)
    ts = np.float32(np.abs(x).max() / np.float32(2688.0))
    blk = np.abs(x).reshape(8, 4, 16).max(axis=2, keepdims=True) / 6.0
    err = np.abs(deq.reshape(8, 4, 16) - x.reshape(8, 4, 16).astype(np.float64))
    # the step at magnitude m/scale <= 6 is at most 2 units of the scale; block scale
    # rounding to E4M3 adds at most 2^-4 relative
    assert np.all(err <= blk * (1 + 2 ** -3) * 1.0 + 1e-6)
    assert float(ts) > 0


# ---------------------------------------------------------------------- router


def pin_select_brute_force(O):
    rng = np.random.default_rng(11)
    shapes = [(16, 4, 2, 4), (12, 3, 2, 3), (12, 4, 1, 2), (16, 2, 1, 5), (9, 3, 3, 4),
              (20, 5, 3, 6), (8, 1, 1, 3)]
    for E, ng, tg, k in shapes:
        for _ in range(40):
            s = O.sigmoid(rng.standard_normal((1, E)))
            bias = rng.normal(0, 0.3, E)
            sel = O.select_experts(s, bias, ng, tg, k)
            want = brute_force_select((s + bias)[0], ng, tg, k)
            assert sorted(sel.ids[0].tolist()) == want, (E, ng, tg, k)


def pin_router_logits(O):
    """l = x W_r^T in fp64: small integers give the exact integer dot products (pins the
    operand order and indexing, H != E), and a single product that needs 25 significant bits,
    (1 + 2^-12)^2 = 1 + 2^-11 + 2^-24, comes out exactly (an fp32 evaluation rounds it)."""
    rng = np.random.default_rng(21)
    x = rng.integers(-4, 5, (3, 5))
    w = rng.integers(-4, 5, (4, 5))
    got = O.router_logits(x.astype(np.float32), w.astype(np.float32))
    want = [[sum(int(x[t, h]) * int(w[e, h]) for h in range(5)) for e in range(4)] for t in range(3)]
    assert got.tolist() == want
    v = np.float32(1 + 2.0 ** -12)
    assert O.router_logits(np.array([[v]]), np.array([[v]]))[0, 0] == 1 + 2.0 ** -11 + 2.0 ** -24


def pin_selection_margins(O):
    """The selection's margins, which the parity checks use to tell near-ties from
    mismatches: group margin = score of the last kept group - score of the first dropped
    group; expert margin = k-th - (k+1)-th biased score among the kept groups' experts; inf
    where nothing is dropped at that level."""
    # hand-worked: groups (0.9, 0.1) (0.8, 0.3) (0.5, 0.45) (0.2, 0.1) score 1.0, 1.1, 0.95,
    # 0.3; groups 1 and 0 kept (margin 1.0 - 0.95); experts 0.9, 0.8 chosen over 0.3
    b = np.array([[0.9, 0.1, 0.8, 0.3, 0.5, 0.45, 0.2, 0.1]])
    sel = O.select_experts(b, np.zeros(8), 4, 2, 2)
    assert sorted(sel.ids[0].tolist()) == [0, 2]
    assert abs(sel.group_margin[0] - 0.05) < 1e-15 and abs(sel.expert_margin[0] - 0.5) < 1e-15
    # every group kept: no group margin; the 2nd and 3rd largest of all eight are 0.8, 0.5
    all_groups = O.select_experts(b, np.zeros(8), 4, 4, 2)
    assert np.isinf(all_groups.group_margin[0]) and abs(all_groups.expert_margin[0] - 0.3) < 1e-15
    all_experts = O.select_experts(b, np.zeros(8), 4, 2, 4)
    assert np.isinf(all_experts.expert_margin[0])
    # brute force on random rows
    rng = np.random.default_rng(22)
    s = rng.uniform(0, 1, (200, 12))
    bias = rng.normal(0, 0.2, 12)
    sel = O.select_experts(s, bias, 4, 2, 3)
    bb = s + bias[None]
    for t in range(200):
        gsc = sorted((sum(sorted(bb[t, 3 * g:3 * g + 3].tolist())[-2:]), g) for g in range(4))[::-1]
        kept = [g for _, g in gsc[:2]]
        cand = sorted((bb[t, e] for g in kept for e in range(3 * g, 3 * g + 3)), reverse=True)
        assert abs(sel.group_margin[t] - (gsc[1][0] - gsc[2][0])) < 1e-12
        assert abs(sel.expert_margin[t] - (cand[2] - cand[3])) < 1e-12
        assert sel.margin[t] == min(sel.group_margin[t], sel.expert_margin[t])


def pin_top_p_margin(O):
    """The adaptive top-p's margin: the distance of the nearest mass-before-rank from the
    threshold p * total, or the score gap across the cut when smaller, over the total; inf
    when nothing can be cut (p outside (0, 1), or one expert)."""
    ids = np.array([[0, 1, 2]])
    # s 0.5, 0.35, 0.15, p 0.7: masses before ranks 1, 2 are 0.5 and 0.85 -> nearest 0.15
    r = O.expert_top_p(np.array([[0.5, 0.35, 0.15]]), ids, 0.7)
    assert r.keep[0].tolist() == [True, True, False] and abs(r.margin[0] - 0.15) < 1e-12
    # s 0.5, 0.26, 0.24, p 0.6: masses 0.5, 0.76 (0.1 away) but the cut separates 0.26 from
    # 0.24 -> 0.02
    r = O.expert_top_p(np.array([[0.5, 0.26, 0.24]]), ids, 0.6)
    assert r.keep[0].tolist() == [True, True, False] and abs(r.margin[0] - 0.02) < 1e-12
    for p in (0.0, 1.0):
        assert np.isinf(O.expert_top_p(np.array([[0.5, 0.26, 0.24]]), ids, p).margin[0])
    assert np.isinf(O.expert_top_p(np.array([[0.5, 0.26, 0.24]]), ids[:, :1], 0.5).margin[0])


def pin_select_special_cases(O):
    rng = np.random.default_rng(5)
    # one group: plain top-k of b, as torch.topk finds it (distinct values)
    s = O.sigmoid(rng.standard_normal((64, 24)))
    bias = rng.normal(0, 0.05, 24)
    sel = O.select_experts(s, bias, 1, 1, 6)
    ref = torch.topk(torch.from_numpy(s + bias), 6, dim=1).indices.numpy()
    assert np.array_equal(np.sort(sel.ids, 1), np.sort(ref, 1))
    # zero bias, one group: top-k of the logits (sigmoid is monotone)
    logits = rng.standard_normal((64, 24))
    sel = O.select_experts(O.sigmoid(logits), np.zeros(24), 1, 1, 5)
    ref = torch.topk(torch.from_numpy(logits), 5, dim=1).indices.numpy()
    assert np.array_equal(np.sort(sel.ids, 1), np.sort(ref, 1))
    # ties: equal scores go to the lower index, among groups and among experts
    b = np.array([[0.5, 0.5, 0.5, 0.5, 0.5, 0.5, 0.5, 0.5]])
    sel = O.select_experts(b, np.zeros(8), 4, 2, 3)
    assert sel.ids[0].tolist() == [0, 1, 2]
    b = np.array([[0.1, 0.9, 0.2, 0.8, 0.9, 0.1, 0.85, 0.85]])   # groups of 2: 1.0, 1.0, 1.0, 1.7
    sel = O.select_experts(b, np.zeros(8), 4, 2, 2)
    assert sorted(sel.ids[0].tolist()) == [1, 6]
    # a group of only negative biased scores still outranks a group of lower ones,
    # and excluded experts never come back (no zero fill)
    b = np.array([[-0.9, -0.8, -0.1, -0.2, -0.95, -0.99]])
    sel = O.select_experts(b, np.zeros(6), 3, 1, 2)
    assert sorted(sel.ids[0].tolist()) == [2, 3]


def pin_routing_weights(O):
    rng = np.random.default_rng(2)
    s = O.sigmoid(rng.standard_normal((50, 16)))
    bias = rng.normal(0, 0.5, 16)
    sel = O.select_experts(s, bias, 4, 2, 4)
    w = O.routing_weights(s, sel.ids, 2.5)
    assert np.allclose(w.sum(1), 2.5, rtol=0, atol=1e-14)
    # weights are proportional to the unbiased scores of the chosen experts
    chosen = np.take_along_axis(s, sel.ids, 1)
    assert np.allclose(w / chosen, (w / chosen)[:, :1], rtol=1e-13)
    # k = 1 gives exactly rsf
    sel1 = O.select_experts(s, bias, 4, 2, 1)
    assert np.all(O.routing_weights(s, sel1.ids, 2.5) == 2.5)


def pin_group_tokens(O):
    rng = np.random.default_rng(4)
    T, k, E = 37, 4, 16
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    counts, offsets, lst = O.group_tokens(ids, E)
    assert counts.sum() == T * k and offsets[-1] == T * k and offsets[0] == 0
    assert np.array_equal(np.diff(offsets), counts)
    for e in range(E):
        ent = lst[offsets[e]:offsets[e + 1]]
        toks, slots = ent // k, ent % k
        assert np.all(np.diff(toks) > 0)
        assert np.all(ids[toks, slots] == e)
    assert sorted(lst.tolist()) == list(range(T * k))


def _top_p_case(O, c, E=8):
    k = len(c["ids"])
    scores = np.full((1, E), 0.01)
    ids = np.asarray([c["ids"]], np.int64)
    scores[0, ids[0]] = c["scores_of_slots"]
    tp = O.expert_top_p(scores, ids, c["p"])
    routed = np.where(tp.keep, ids, -1)
    w = O.routing_weights(scores, routed, 2.5)
    return tp, routed, w, k


def pin_expert_top_p_hand(O):
    """Hand-worked adaptive top-p cases (tests/golden/hand_expert_top_p.json)."""
    with open(os.path.join(GOLDEN, "hand_expert_top_p.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        tp, routed, w, k = _top_p_case(O, c)
        assert tp.keep[0].tolist() == c["keep"], (c["p"], tp.keep[0].tolist())
        assert np.allclose(w[0], c["weights"], rtol=1e-15, atol=0), (c["p"], w[0])


def pin_expert_top_p_invariants(O):
    """On random scores: the kept mass reaches p * total and dropping the smallest kept
    score would fall below it (shortest prefix); kept scores are the largest ones; the
    weights are 0 on dropped slots, sum to rsf and stay proportional to s; grouping skips
    dropped slots."""
    rng = np.random.default_rng(11)
    E, k = 32, 8
    for p in (0.3, 0.7, 0.9):
        s = O.sigmoid(rng.standard_normal((40, E)))
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(40)])
        tp = O.expert_top_p(s, ids, p)
        routed = np.where(tp.keep, ids, -1)
        w = O.routing_weights(s, routed, 2.5)
        for t in range(40):
            sel = s[t, ids[t]]
            kept = sel[tp.keep[t]]
            assert kept.sum() >= p * sel.sum() - 1e-15
            assert kept.sum() - kept.min() < p * sel.sum()
            if (~tp.keep[t]).any():
                assert kept.min() >= sel[~tp.keep[t]].max()
            assert np.all(w[t][~tp.keep[t]] == 0)
            assert abs(w[t].sum() - 2.5) < 1e-13
            ratio = w[t][tp.keep[t]] / kept
            assert np.allclose(ratio, ratio[0], rtol=1e-13)
        counts, offsets, lst = O.group_tokens(routed, E)
        assert offsets[-1] == tp.keep.sum() == lst.size
        assert np.all(routed.ravel()[lst] >= 0)


def pin_int_row_formats(O):
    """Per-row integer formats, hand-decoded bytes: int8 one per byte, int4 element 2j in
    the low nibble, int2 element 4j + i in bits 2i..2i+1, all two's complement; the row
    scale multiplies every element of its row."""
    assert O.decode_int_row(np.array([[0x00, 0x7F, 0x80, 0xFF]], np.uint8), 8).tolist() == [[0, 127, -128, -1]]
    assert O.decode_int_row(np.array([[0x8F, 0x71]], np.uint8), 4).tolist() == [[-1, -8, 1, 7]]
    assert O.decode_int_row(np.array([[0xE4, 0x1B]], np.uint8), 2).tolist() == [[0, 1, -2, -1, -1, -2, 1, 0]]
    w = O.dequant_int_row(np.array([[0xE4], [0x1B]], np.uint8), np.array([[0.5], [4.0]], np.float32), 2)
    assert w.tolist() == [[0.0, 0.5, -1.0, -0.5], [-4.0, -8.0, 4.0, 0.0]]


def pin_int_row_roundtrip(O):
    """The generator's per-row quantiser decoded by the oracle stays within half a step
    (|w - code * scale| <= scale / 2; the largest |w| of a row maps to qmax exactly)."""
    from synth.layer import quantize_int_row
    rng = np.random.default_rng(13)
    w = rng.normal(0, 0.05, (16, 128)).astype(np.float32)
    for bits in (8, 4, 2):
        codes, scale = quantize_int_row(w, bits)
        deq = O.dequant_int_row(codes, scale, bits)
        assert np.all(np.abs(deq - w) <= scale.astype(np.float64) / 2 * (1 + 1e-6))
        qmax = (1 << (bits - 1)) - 1
        assert np.all(np.abs(O.decode_int_row(codes, bits)).max(axis=1) == qmax)


def pin_q8_0_activation(O):
    """Q8_0 activations, hand-worked: exact multiples of the block step come back exactly;
    halfway quotients round to even; the block step is the fp16 value of amax / 127
    (amax 1 gives d = 516 / 65536, so 1 -> 127 d = 0.99993896484375 and 0.5 -> 64 d =
    0.50390625); an all-zero block stays zero; blocks are 32 wide."""
    n = np.arange(-16, 16, dtype=np.float64)
    n[0] = -127.0
    a = (n / 16.0)[None, :]
    assert np.array_equal(O.quantize_q8_0_activation(a), a)
    b = np.zeros((1, 32))
    b[0, :4] = [127.0, 2.5, 3.5, -0.5]
    assert O.quantize_q8_0_activation(b)[0, :4].tolist() == [127.0, 2.0, 4.0, 0.0]
    c = np.zeros((1, 64))
    c[0, :2] = [1.0, 0.5]
    got = O.quantize_q8_0_activation(c)
    assert got[0, 0] == 0.99993896484375 and got[0, 1] == 0.50390625
    assert not got[0, 2:].any()


def pin_q8_0_layer_composition(O):
    """Q8_0 in the whole layer, recomposed token by token from the pinned parts: x quantised
    before every expert's gate/up (routed and shared), each expert's h quantised before its
    down projection, the weighted combine, the shared expert added with weight 1."""
    from dataclasses import replace

    from synth import LAYERS, make_layer, make_x
    spec = replace(LAYERS["tiny"], name="tiny_int4row_q8", weight_format="int4_row",
                   shared_format="int4_row", act_quant="q8_0")
    layer = O.Layer.from_spec(spec, make_layer(spec))
    x = make_x(spec, 5, 0)
    ref = layer.forward(x)
    I = spec.inter
    xq = O.quantize_q8_0_activation(x)
    got = np.zeros_like(ref.out)

    def ffn(w_gu, w_d, xt):
        gu = w_gu @ xt
        h = O.silu(gu[:I]) * gu[I:]
        return w_d @ O.quantize_q8_0_activation(h[None, :])[0]

    sh_gu, sh_d = layer.shared_expert()
    for t in range(x.shape[0]):
        for j in range(spec.top_k):
            e = int(ref.ids[t, j])
            got[t] += ref.weights[t, j] * ffn(layer.routed_gu(e), layer.routed_d(e), xq[t])
        got[t] += ffn(sh_gu, sh_d, xq[t])
    assert np.allclose(got, ref.out, rtol=1e-12, atol=1e-14)
    # and the quantisation matters here (the unquantised layer differs)
    plain = O.Layer.from_spec(replace(spec, act_quant="none"), make_layer(spec)).forward(x).out
    assert not np.allclose(plain, ref.out, rtol=1e-6, atol=0)


def pin_nvfp4_layer_composition(O):
    """NVFP4 in the whole layer, recomposed token by token from the pinned parts: x quantised
    once for the call (one tensor scale over every token), each routed expert's gate/up on
    those rows, all routed h rows of the call quantised together (one h tensor scale), the
    down projection, the weighted combine, and the bf16 shared expert on the unquantised x.
    Token 1 is rescaled to three times token 0's amax, so a tensor scale per token would move
    token 0's block scales through E4M3 rounding: checked to change the output."""
    from dataclasses import replace

    from synth import LAYERS, make_layer, make_x
    spec = replace(LAYERS["tiny"], name="tiny_nvfp4_f32", weight_format="nvfp4", shared_format="bf16")
    layer = O.Layer.from_spec(spec, make_layer(spec))
    x = make_x(spec, 4, 0)
    a0, a1 = np.abs(x[0]).max(), np.abs(x[1]).max()
    x[1] = (x[1] * np.float32(3.0 * a0 / a1)).astype(np.float32)
    ref = layer.forward(x)
    I = spec.inter

    def compose(xq):
        hs = {}
        for e in range(spec.n_experts):
            ent = ref.entries[ref.offsets[e]:ref.offsets[e + 1]]
            if ent.size:
                gu = xq[ent // spec.top_k] @ layer.routed_gu(e).T
                hs[e] = (ent, O.silu(gu[:, :I]) * gu[:, I:])
        out = np.zeros_like(ref.out)
        for e, (ent, h) in O.quantize_routed_h(hs).items():
            for r, y in zip(ent, h @ layer.routed_d(e).T):
                t, j = divmod(int(r), spec.top_k)
                out[t] += ref.weights[t, j] * y
        sh_gu, sh_d = layer.shared_expert()
        gu = x.astype(np.float64) @ sh_gu.T
        return out + (O.silu(gu[:, :I]) * gu[:, I:]) @ sh_d.T

    got = compose(O.quantize_nvfp4_activation(x))
    assert np.allclose(got, ref.out, rtol=1e-12, atol=1e-14)
    per_token = compose(np.vstack([O.quantize_nvfp4_activation(x[t:t + 1]) for t in range(4)]))
    assert not np.allclose(per_token[0], ref.out[0], rtol=1e-6, atol=0)


def pin_top_p_layer_composition(O):
    """The adaptive top-p inside the layer: the routed ids are the selection cut by
    expert_top_p (dropped slots -1, some dropped here), the weights are renormalised over the
    kept slots, and the output equals the forward re-run on those ids."""
    from dataclasses import replace

    from synth import LAYERS, make_layer, make_x
    spec = replace(LAYERS["tiny"], expert_top_p=0.6)
    arrays = make_layer(spec)
    layer = O.Layer.from_spec(spec, arrays)
    x = make_x(spec, 12, 1)
    ref = layer.forward(x)
    scores, sel = layer.route(layer.widen_x(x))
    keep = O.expert_top_p(scores, sel.ids, 0.6).keep
    assert (~keep).any()
    assert np.array_equal(ref.ids, np.where(keep, sel.ids, -1))
    assert np.allclose(ref.weights.sum(axis=1), spec.rsf, atol=1e-12)
    assert np.all(ref.weights[~keep] == 0)
    full = O.Layer.from_spec(replace(spec, expert_top_p=0.0), arrays)
    assert np.allclose(full.forward(x, ids=ref.ids).out, ref.out, rtol=1e-13, atol=1e-15)


# ------------------------------------------------------------------- expert FFN


def pin_expert_ffn_torch(O):
    rng = np.random.default_rng(9)
    w_gu = rng.normal(0, 0.3, (2 * 48, 64))
    w_d = rng.normal(0, 0.3, (64, 48))
    x = rng.standard_normal((5, 64))
    h = O.swiglu_hidden(w_gu, x)
    y = O.down_proj(w_d, h)
    tx, tgu, td = (torch.from_numpy(a) for a in (x, w_gu, w_d))
    gu = torch.nn.functional.linear(tx, tgu)
    th = torch.nn.functional.silu(gu[:, :48]) * gu[:, 48:]
    ty = torch.nn.functional.linear(th, td)
    assert torch.allclose(torch.from_numpy(h), th, rtol=1e-13, atol=1e-15)
    assert torch.allclose(torch.from_numpy(y), ty, rtol=1e-12, atol=1e-14)


def pin_hand_two_expert(O):
    s0, s1 = sigmoid_scalar(0.25), sigmoid_scalar(-1.0)
    h_e0 = silu_scalar(0.75) * 0.625
    h_e1 = silu_scalar(4.0) * 2.0
    h_sh = silu_scalar(1.0) * 3.0
    # k = 2: both experts, weights from the unbiased scores
    layer, x = hand_layer(O, "k2")
    ref = layer.forward(x)
    w0, w1 = s0 / (s0 + s1) * 2.5, s1 / (s0 + s1) * 2.5
    expect = np.zeros(32)
    expect[0] = w0 * 2 * h_e0 + w1 * h_e1
    expect[5] = w0 * -3 * h_e0
    expect[7] = w1 * 0.875 * h_e1
    expect[1] = -2 * h_sh
    assert np.allclose(ref.out[0], expect, rtol=1e-12, atol=1e-14), (ref.out[0][:8], expect[:8])
    # k = 2 with a bias: both experts are chosen all the same, and noaux_tc's bias only
    # selects, so the weights (per expert) and the output are those of the unbiased case
    layer, x = hand_layer(O, "k2_bias")
    ref_b = layer.forward(x)
    assert sorted(ref_b.ids[0].tolist()) == [0, 1]
    w_of = dict(zip(ref_b.ids[0].tolist(), ref_b.weights[0].tolist()))
    assert np.allclose([w_of[0], w_of[1]], [w0, w1], rtol=1e-14, atol=0), (w_of, w0, w1)
    assert np.allclose(ref_b.out[0], expect, rtol=1e-12, atol=1e-14), (ref_b.out[0][:8], expect[:8])
    # k = 1 with a bias that flips the choice to expert 1; its weight is exactly rsf
    layer, x = hand_layer(O, "k1")
    ref = layer.forward(x)
    assert ref.ids.tolist() == [[1]]
    expect = np.zeros(32)
    expect[0] = 2.5 * h_e1
    expect[7] = 2.5 * 0.875 * h_e1
    expect[1] = -2 * h_sh
    assert np.allclose(ref.out[0], expect, rtol=1e-12, atol=1e-14), (ref.out[0][:8], expect[:8])


def pin_identity_activation_exact(O):
    """The hand-worked layer with the SiLU bypassed: at k = 1 the weight is exactly rsf and
    every product is a small dyadic number, so the output is known exactly (gate 4, up 2
    for expert 1; gate 1, up 3 for the shared expert)."""
    layer, x = hand_layer(O, "k1")
    ref = layer.forward(x, activation="identity")
    assert ref.ids.tolist() == [[1]]
    expect = np.zeros(32)
    expect[0] = 2.5 * (4.0 * 2.0)
    expect[7] = 2.5 * 0.875 * (4.0 * 2.0)
    expect[1] = -2 * (1.0 * 3.0)
    assert np.array_equal(ref.out[0], expect), (ref.out[0][:8], expect[:8])


def pin_hand_nvfp4_layer(O):
    """The hand-worked NVFP4 layer: one h tensor scale over every routed h row of the call,
    and the bf16 shared expert fed the unquantised x (closed form in the fixture)."""
    layer, x = hand_nvfp4_layer(O)
    ref = layer.forward(x, activation="identity")
    assert sorted(ref.ids[0].tolist()) == [0, 1]
    ts_x = float(np.float32(6.0) / np.float32(2688.0))
    r = 448.0 * ts_x
    ts_h = float(np.float32(np.float32(8.0 * r * r) / np.float32(2688.0)))
    h0_q, h1_q = 6.0 * 448.0 * ts_h, 6.0 * 256.0 * ts_h
    s0, s1 = sigmoid_scalar(0.25), sigmoid_scalar(-1.0)
    w0, w1 = s0 / (s0 + s1) * 2.5, s1 / (s0 + s1) * 2.5
    expect = np.zeros(32)
    expect[0] = w0 * h0_q + w1 * 0.5 * h1_q
    expect[3] = w0 * -0.5 * h0_q
    expect[5] = w1 * 2.0 * h1_q
    expect[7] = 0.30078125 * 2.0
    assert np.allclose(ref.out[0], expect, rtol=1e-12, atol=1e-15), (ref.out[0][:8], expect[:8])


def pin_widen_bf16(O):
    """Every bf16 bit pattern widens to the value torch's bfloat16 -> float64 gives."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        got = O.widen_bf16(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def pin_layer_invariants(O, spec, arrays, x):
    """Token permutation commutes with the layer; the routing weights sum to rsf;
    doubling every routed W_d scale doubles the routed part of the output."""
    layer = O.Layer.from_spec(spec, arrays)
    ref = layer.forward(x)
    perm = np.random.default_rng(1).permutation(x.shape[0])
    ref_p = layer.forward(x[perm])
    assert np.allclose(ref_p.out, ref.out[perm], rtol=1e-12, atol=1e-15)
    assert np.allclose(ref.weights.sum(1), spec.rsf, atol=1e-12)
    a2 = dict(arrays)
    a2["d_scales"] = (arrays["d_scales"].astype(np.float32) * 2).astype(arrays["d_scales"].dtype)
    ref2 = O.Layer.from_spec(spec, a2).forward(x)
    a0 = dict(arrays)
    a0["d_scales"] = np.zeros_like(arrays["d_scales"])
    shared_only = O.Layer.from_spec(spec, a0).forward(x).out
    assert np.allclose(ref2.out - shared_only, 2 * (ref.out - shared_only), rtol=1e-11, atol=1e-14)


ALL_PINS = [pin_decode_int4, pin_decode_e4m3, pin_decode_e2m1, pin_dequant_int4_g32,
            pin_dequant_nvfp4, pin_nvfp4_rounding, pin_nvfp4_activation, pin_select_brute_force,
            pin_select_special_cases, pin_routing_weights, pin_group_tokens,
            pin_expert_ffn_torch, pin_hand_two_expert, pin_identity_activation_exact,
            pin_hand_nvfp4_layer, pin_widen_bf16, pin_expert_top_p_hand,
            pin_expert_top_p_invariants, pin_int_row_formats, pin_int_row_roundtrip,
            pin_q8_0_activation, pin_q8_0_layer_composition, pin_top_p_layer_composition,
            pin_router_logits, pin_selection_margins, pin_top_p_margin,
            pin_nvfp4_layer_composition]
