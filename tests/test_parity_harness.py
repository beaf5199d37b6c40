"""The parity checks themselves, on the CPU: results derived from the oracle pass them,
and the same results with a typical GPU mistake planted (a wrong expert, permuted or
unscaled weights, a broken entry list, a missing shared expert, swapped tokens, a small
bias in the output) fail them. A check that missed one of these would let the GPU tests
pass a broken kernel."""

import numpy as np
import pytest

from oracle.moe_oracle import Layer
from synth import LAYERS, make_layer, make_x
from tests.parity import NEAR_TIE, check_out, check_routing, valid_selection

SPEC = LAYERS["tiny"]     # H 256, I 128, E 16 in 4 groups, top-2 groups, k 4


@pytest.fixture(scope="module")
def case():
    arrays = make_layer(SPEC)
    oracle = Layer.from_spec(SPEC, arrays)
    x = make_x(SPEC, 24, 7)
    return arrays, oracle, x, oracle.forward(x)


def gpu_view(ref):
    """The routing as moe_layer_get_routing returns it, taken from the oracle."""
    return {"ids": ref.ids.astype(np.int32).copy(), "weights": ref.weights.astype(np.float32).copy(),
            "offsets": ref.offsets.astype(np.int32).copy(), "entries": ref.entries.astype(np.int32).copy()}


def routing_ok(arrays, ref, got):
    try:
        check_routing(ref, got, bias=arrays["bias"], n_group=SPEC.n_group, topk_group=SPEC.topk_group,
                      top_k=SPEC.top_k, n_experts=SPEC.n_experts)
        return True
    except AssertionError:
        return False


def out_ok(ref_out, got):
    try:
        check_out(ref_out, got)
        return True
    except AssertionError:
        return False


def clear_token(ref):
    """A token whose selection is far from any tie."""
    return int(np.argmax(ref.margin))


def test_oracle_results_pass(case):
    arrays, _, _, ref = case
    assert routing_ok(arrays, ref, gpu_view(ref))
    assert out_ok(ref.out, ref.out.astype(np.float32))
    # fp16-level noise on every element passes
    rng = np.random.default_rng(0)
    assert out_ok(ref.out, ref.out * (1 + 5e-4 * rng.standard_normal(ref.out.shape)))


def test_wrong_expert_is_caught(case):
    arrays, _, _, ref = case
    got = gpu_view(ref)
    t = clear_token(ref)
    assert ref.margin[t] > NEAR_TIE
    unused = [e for e in range(SPEC.n_experts) if e not in got["ids"][t]]
    got["ids"][t, -1] = unused[0]
    assert not routing_ok(arrays, ref, got)


def test_weight_mistakes_are_caught(case):
    arrays, _, _, ref = case
    got = gpu_view(ref)
    got["weights"] = np.roll(got["weights"], 1, axis=1)          # weight of the wrong slot
    assert not routing_ok(arrays, ref, got)
    got = gpu_view(ref)
    got["weights"] = got["weights"] / np.float32(SPEC.rsf)        # rsf forgotten
    assert not routing_ok(arrays, ref, got)
    got = gpu_view(ref)
    got["weights"][3, 0] *= np.float32(1 + 1e-4)                  # one weight off by 1e-4
    assert not routing_ok(arrays, ref, got)


def test_entry_list_mistakes_are_caught(case):
    arrays, _, _, ref = case
    off = ref.offsets
    e = int(np.argmax(np.diff(off)))                              # the busiest expert
    assert off[e + 1] - off[e] >= 2
    got = gpu_view(ref)
    got["entries"][off[e]:off[e + 1]] = got["entries"][off[e]:off[e + 1]][::-1]   # descending tokens
    assert not routing_ok(arrays, ref, got)
    got = gpu_view(ref)
    r = int(got["entries"][off[e]])
    got["entries"][off[e]] = (r // SPEC.top_k) * SPEC.top_k + (r % SPEC.top_k + 1) % SPEC.top_k  # wrong slot
    assert not routing_ok(arrays, ref, got)
    got = gpu_view(ref)
    got["offsets"][-1] -= 1                                       # an entry missing from the count
    assert not routing_ok(arrays, ref, got)
    got = gpu_view(ref)
    got["offsets"][e + 1] += 1                                    # an entry moved to the next expert
    assert not routing_ok(arrays, ref, got)


def test_output_mistakes_are_caught(case):
    _, oracle, x, ref = case
    sh_gu, sh_d = oracle.shared_expert()
    x64 = oracle.widen_x(x)
    gu = x64 @ sh_gu.T
    I = SPEC.inter
    shared = (gu[:, :I] / (1 + np.exp(-gu[:, :I])) * gu[:, I:]) @ sh_d.T
    assert not out_ok(ref.out, ref.out - shared)                  # shared expert missing
    got = ref.out.copy()
    got[[0, 1]] = got[[1, 0]]                                     # two tokens swapped
    assert not out_ok(ref.out, got)
    got = ref.out.copy()
    got[5] = 0                                                    # one token never written
    assert not out_ok(ref.out, got)
    assert not out_ok(ref.out, ref.out * 1.01)                    # 1 % scale error
    got = ref.out.copy()
    got[:, 7] += 0.02 * np.abs(ref.out).max()                     # one column biased by 2 %
    assert not out_ok(ref.out, got)


def test_valid_selection_accepts_ties_and_rejects_invalid_sets():
    # groups of 4: (9, 8, 1, 1) (7, 6, 1, 1) (2, 2, 1, 1) (0, 0, 0, 0): kept groups 0 and 1
    b = np.array([9, 8, 1, 1, 7, 6, 1, 1, 2, 2, 1, 1, 0, 0, 0, 0], np.float64)
    assert valid_selection(b, [0, 1, 4, 5], 4, 2, 1e-9)
    assert not valid_selection(b, [0, 1, 4, 8], 4, 2, 1e-9)       # an expert of a dropped group
    assert not valid_selection(b, [0, 1, 4, 2], 4, 2, 1e-9)       # 1 chosen over 6
    assert not valid_selection(b, [0, 1, 4, 4], 4, 2, 1e-9)       # a repeated expert
    # all four from group 0, although group 1 is kept and holds 7 and 6
    assert not valid_selection(b, [0, 1, 2, 3], 4, 2, 1e-9)
    # an exact tie between 6 and a second 6 in another kept group may go either way
    b2 = b.copy()
    b2[1] = 6.0
    assert valid_selection(b2, [0, 1, 4, 5], 4, 2, 1e-9) and valid_selection(b2, [0, 4, 5, 1], 4, 2, 1e-9)


@pytest.mark.parametrize("E,n_group,topk_group,k", [(16, 4, 2, 4), (32, 8, 4, 8), (64, 8, 3, 6)])
def test_valid_selection_holds_for_selections_near_the_scores(E, n_group, topk_group, k):
    """Scores on a coarse grid (so that exact ties between experts and between groups are
    common), perturbed by at most tol / 4: the exact selection on the perturbed scores is a
    valid selection of the unperturbed ones."""
    from oracle.moe_oracle import select_experts
    rng = np.random.default_rng(E + k)
    tol = 1e-5
    for _ in range(300):
        b = rng.integers(0, 6, E) / 8.0
        bp = b + rng.uniform(-tol / 4, tol / 4, E)
        ids = select_experts(bp[None], np.zeros(E), n_group, topk_group, k).ids[0]
        assert valid_selection(b, ids, n_group, topk_group, tol), (b, ids)


@pytest.mark.parametrize("E,n_group,topk_group,k", [(16, 4, 2, 4), (32, 8, 4, 8)])
def test_valid_selection_rejects_clearly_worse_sets(E, n_group, topk_group, k):
    """With distinct scores far from any tie, giving up a chosen expert for a lower one of a
    kept group, or for any expert of a dropped group, is invalid."""
    from oracle.moe_oracle import select_experts
    rng = np.random.default_rng(3 * E + k)
    G = E // n_group
    checked = 0
    for _ in range(300):
        b = rng.permutation(E) / E              # distinct, at least 1/E apart
        sel = select_experts(b[None], np.zeros(E), n_group, topk_group, k)
        ids = sel.ids[0].tolist()
        assert valid_selection(b, ids, n_group, topk_group, 1e-5)
        gs = np.sort(b.reshape(n_group, G), axis=1)[:, -2:].sum(1)
        kept = set(np.argsort(-gs, kind="stable")[:topk_group].tolist())
        lower = [e for e in range(E) if e // G in kept and e not in ids]
        dropped = [e for e in range(E) if e // G not in kept]
        for bad in (lower[:1] + dropped[:1]):
            worse = ids[:-1] + [bad] if bad != ids[-1] else ids[1:] + [bad]
            if sorted(worse) == sorted(ids):
                continue
            assert not valid_selection(b, worse, n_group, topk_group, 1e-5), (b, ids, worse)
            checked += 1
    assert checked > 300
