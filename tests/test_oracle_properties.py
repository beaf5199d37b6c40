"""Property tests of the oracle's routing on random shapes, with ties (CPU).

Scores are drawn from a grid of multiples of 1/64, so exact ties between experts and
between groups are frequent and every sum below is exact in fp64. Each property is checked
against an independent formulation:
- selection: exhaustive search over all group subsets, then all expert subsets, for the
  largest summed score, with ties going to the lexicographically smallest index set (the
  oracle's rule, lower index first, stated for subsets);
- slot order: descending biased score, lower id first;
- adaptive top-p: the smallest number m of top-ranked experts whose score mass reaches
  p times the total (ranked by score, lower id first);
- grouping: a sort of all routed (expert, token, slot) triples.
"""

from itertools import combinations

import numpy as np
from hypothesis import given, settings
from hypothesis import strategies as st

from oracle import moe_oracle as O

GRID = st.integers(-64, 64).map(lambda i: i / 64.0)
SETTINGS = settings(max_examples=300, deadline=None, derandomize=True)


@st.composite
def routing_case(draw):
    n_group = draw(st.integers(1, 4))
    G = draw(st.integers(2, 4))
    E = n_group * G
    topk_group = draw(st.integers(1, n_group))
    top_k = draw(st.integers(1, topk_group * G))
    b = np.array(draw(st.lists(GRID, min_size=E, max_size=E)))
    return b, n_group, topk_group, top_k


def best_subset(values, size):
    """Index set of the given size with the largest sum; ties: lexicographically smallest."""
    return min(combinations(range(len(values)), size), key=lambda c: (-sum(values[i] for i in c), c))


@SETTINGS
@given(routing_case())
def test_selection_is_the_best_subset_with_lower_index_ties(case):
    b, n_group, topk_group, top_k = case
    G = b.size // n_group
    gscore = [sum(sorted(b[g * G:(g + 1) * G])[-2:]) for g in range(n_group)]
    groups = best_subset(gscore, topk_group)
    cand = [e for g in sorted(groups) for e in range(g * G, (g + 1) * G)]
    pick = best_subset([b[e] for e in cand], top_k)
    want = sorted(cand[i] for i in pick)
    sel = O.select_experts(b[None] - 0.0, np.zeros(b.size), n_group, topk_group, top_k)
    ids = sel.ids[0].tolist()
    assert sorted(ids) == want
    assert ids == sorted(ids, key=lambda e: (-b[e], e))          # slot order
    assert np.all(sel.margin >= 0)


@SETTINGS
@given(st.integers(2, 8).flatmap(lambda k: st.tuples(
    st.just(k), st.lists(st.integers(1, 64).map(lambda i: i / 64.0), min_size=k, max_size=k),
    st.sampled_from([0.125, 0.25, 0.5, 0.625, 0.75, 0.875]))))
def test_top_p_keeps_the_shortest_ranked_prefix_reaching_p(case):
    k, scores, p = case
    s = np.array(scores)[None]
    ids = np.arange(k)[None]
    keep = O.expert_top_p(s, ids, p).keep[0]
    order = sorted(range(k), key=lambda j: (-s[0, j], j))
    total = sum(scores)
    m = next(m for m in range(1, k + 1) if sum(s[0, j] for j in order[:m]) >= p * total)
    assert sorted(np.flatnonzero(keep).tolist()) == sorted(order[:m])


@SETTINGS
@given(st.integers(1, 6).flatmap(lambda T: st.integers(1, 4).flatmap(lambda k: st.integers(k, 8).flatmap(
    lambda E: st.tuples(st.just(E), st.lists(st.lists(st.integers(-1, E - 1), min_size=k, max_size=k),
                                              min_size=T, max_size=T))))))
def test_grouping_is_a_sort_of_the_routed_triples(case):
    E, rows = case
    ids = np.array(rows)
    T, k = ids.shape
    counts, offsets, entries = O.group_tokens(ids, E)
    triples = sorted((int(ids[t, j]), t, j) for t in range(T) for j in range(k) if ids[t, j] >= 0)
    assert entries.tolist() == [t * k + j for _, t, j in triples]
    assert counts.tolist() == [sum(1 for e, _, _ in triples if e == x) for x in range(E)]
    assert offsets.tolist() == [0] + np.cumsum(counts).tolist()
