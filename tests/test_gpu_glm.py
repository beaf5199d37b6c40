"""GPU parity on the GLM-5.2-shaped layer (H=6144, I=2048, E=256 + 1 shared, k=8,
n_group=8, topk_group=4, int4 with fp16 scales per 32): decode at T=1, T=4 and T=32
(unbiased router) and prefill at T=2048 (bias N(0, 0.5)). Routing is checked for every
token; outputs for every token up to T=32, and at T=2048 for 320 tokens that include every
256-row chunk boundary of the most loaded expert and every token of the experts that
received a single token."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle.moe_oracle import Layer
from synth import LAYERS, make_layer, make_x, with_bias_of
from tests.gpu_util import empty_out, out_to_host, x_to_device
from tests.parity import check_out, check_routing


@pytest.fixture(scope="module")
def glm_base():
    return make_layer(LAYERS["glm52"])


_layers = {}


def get_layer(name, base):
    import quantized_moe_noaux_b300 as moe
    if name not in _layers:
        spec = LAYERS[name]
        arrays = base if name == "glm52" else with_bias_of(base, spec)
        _layers[name] = (spec, arrays, moe.MoeLayer.from_spec(spec, arrays, max_tokens=2048),
                         Layer.from_spec(spec, arrays))
    return _layers[name]


def check(name, base, T, step, sample=None, path=None):
    spec, arrays, layer, oracle = get_layer(name, base)
    if path is not None:
        layer.set_path(path)
    x = make_x(spec, T, step)
    out = empty_out(T, spec.hidden, spec.act_dtype)
    layer.forward(x_to_device(x, spec.act_dtype), out)
    torch.cuda.synchronize()
    assert layer.status() == 0
    got = layer.routing(T)
    x64 = oracle.widen_x(x)
    scores, sel = oracle.route(x64)
    from oracle.moe_oracle import routing_weights, group_tokens

    class R:  # routing-only oracle result for all T tokens
        pass
    r = R()
    r.ids, r.scores, r.margin = sel.ids, scores, sel.margin
    r.weights = routing_weights(scores, sel.ids, spec.rsf)
    r.counts, r.offsets, r.entries = group_tokens(sel.ids, spec.n_experts)
    rep = check_routing(r, got, bias=arrays["bias"], n_group=spec.n_group,
                        topk_group=spec.topk_group, top_k=spec.top_k, n_experts=spec.n_experts)
    toks = np.arange(T) if sample is None else np.asarray(sample)
    ids = got["ids"] if rep["mismatch"] else None
    ref = oracle.forward(x, ids=ids, tokens=toks)
    errs = check_out(ref.out[toks], out_to_host(out)[toks])
    counts = np.diff(got["offsets"])
    return errs, counts, rep


@pytest.mark.parametrize("step", [0, 1, 2])
def test_decode_t1(glm_base, step):
    check("glm52", glm_base, 1, step)


def test_decode_t4(glm_base):
    check("glm52_unbiased", glm_base, 4, 0)


def test_decode_t32(glm_base):
    check("glm52_unbiased", glm_base, 32, 0)


@pytest.mark.parametrize("T", [3, 5])
def test_mtp_verify_batch(glm_base, T):
    """MTP draft-verify forward (the accepted position and T - 1 draft positions in one
    batch-union call) through the fused decode kernel: every position's routing and output;
    the experts read once for all positions are the union of the positions' selections."""
    import quantized_moe_noaux_b300 as moe
    check("glm52", glm_base, T, 40 + T, path=moe.PATH_GEMV)
    spec, _, layer, _ = get_layer("glm52", glm_base)
    layer.set_path(moe.PATH_AUTO)
    got = layer.routing(T)
    union = set(got["ids"].ravel().tolist())
    assert int(np.count_nonzero(np.diff(got["offsets"]))) == len(union)


def prefill_sample(routing, top_k, T, n=320, seed=0):
    """Tokens whose outputs are compared at T=2048: the first and last token of every
    256-row chunk of the most loaded expert's entry list (the grouped GEMM's tile
    boundaries), every token of the experts that got one token, then seeded random tokens
    up to n."""
    off, ent = routing["offsets"], routing["entries"]
    counts = np.diff(off)
    e_max = int(np.argmax(counts))
    toks = ent[off[e_max]:off[e_max + 1]] // top_k
    pick = set()
    for c0 in range(0, len(toks), 256):
        pick.add(int(toks[c0]))
        pick.add(int(toks[min(c0 + 255, len(toks) - 1)]))
    for e in np.nonzero(counts == 1)[0]:
        pick.add(int(ent[off[e]] // top_k))
    rng = np.random.default_rng(seed)
    for t in rng.permutation(T):
        if len(pick) >= n:
            break
        pick.add(int(t))
    return np.array(sorted(pick)), e_max, int(counts[e_max])


def test_prefill_t2048(glm_base):
    spec, arrays, layer, oracle = get_layer("glm52_skewed", glm_base)
    # routing first, to choose the compared tokens from the GPU's own entry lists
    x = make_x(spec, 2048, 0)
    out = empty_out(2048, spec.hidden, spec.act_dtype)
    layer.forward(x_to_device(x, spec.act_dtype), out)
    torch.cuda.synchronize()
    sample, e_max, n_max = prefill_sample(layer.routing(2048), spec.top_k, 2048)
    assert n_max > 3 * 256                                  # the heavy expert spans several chunks
    errs, counts, rep = check("glm52_skewed", glm_base, 2048, 0, sample=sample)
    assert counts.sum() == 2048 * 8
    assert counts.max() > 4 * counts[counts > 0].mean()    # the wide bias skews the load


def test_decode_t1_bench_steps_routing(glm_base):
    """The bench's default decode workload (seeds 10..1009, one token per step, the timed
    steps of `bench.py` with its defaults) through the fused kernel: every step's
    selection, weights and the kernel's own grouping (offsets and entries) against the
    oracle (near-tie rule); outputs for three of the steps."""
    spec, arrays, layer, oracle = get_layer("glm52", glm_base)
    from oracle.moe_oracle import group_tokens, routing_weights
    seeds = list(range(10, 1010))
    samples = {0: None, 499: None, 999: None}          # step index -> output row
    xs = np.concatenate([make_x(spec, 1, s) for s in seeds])
    k = spec.top_k
    out = empty_out(1, spec.hidden, spec.act_dtype)
    got_steps = []
    for i in range(len(seeds)):
        layer.forward(x_to_device(xs[i:i + 1], spec.act_dtype), out)
        got_steps.append(layer.routing(1))
        if i in samples:
            samples[i] = out_to_host(out)[0]
    torch.cuda.synchronize()
    assert layer.status() == 0
    scores, sel = oracle.route(oracle.widen_x(xs))

    class R:  # routing-only oracle result of one step
        pass
    mismatch = set()
    for i, got in enumerate(got_steps):
        ref = R()
        ref.ids, ref.scores, ref.margin = sel.ids[i:i + 1], scores[i:i + 1], sel.margin[i:i + 1]
        ref.weights = routing_weights(ref.scores, ref.ids, spec.rsf)
        ref.counts, ref.offsets, ref.entries = group_tokens(ref.ids, spec.n_experts)
        rep = check_routing(ref, got, bias=arrays["bias"], n_group=spec.n_group,
                            topk_group=spec.topk_group, top_k=k, n_experts=spec.n_experts)
        if rep["mismatch"]:
            mismatch.add(i)
    for i, row in samples.items():
        use = got_steps[i]["ids"] if i in mismatch else None
        o = oracle.forward(xs[i:i + 1], ids=use)
        check_out(o.out, row[None])
