"""Comparison of the CUDA layer against the fp64 oracle.

Contract (per token t):
* expert ids: the chosen set must equal the oracle's whenever the oracle's selection
  margin exceeds NEAR_TIE (1e-5, five times the fp32 logit error); within NEAR_TIE the
  GPU's set must still be a valid top-k under the fp64 scores to within NEAR_TIE (with the
  adaptive top-p: a non-empty kept set; its margin is the distance of the cut from its
  threshold), and the outputs of such tokens are compared with the oracle re-run on the
  GPU's ids; dropped slots read id -1 and weight 0;
* entry lists: per expert, the tokens in ascending order and each entry's slot pointing
  at that expert in the GPU's own ids (slot order is not part of the contract);
* combine weights: relative error <= 1e-5 against the oracle's weight of the same expert;
* outputs: relative L2 error <= 2e-3 and max |err| <= 1e-2 * max |ref|.
"""

from __future__ import annotations

import numpy as np

NEAR_TIE = 1e-5
REL_L2 = 2e-3
MAX_REL = 1e-2


def valid_selection(b: np.ndarray, ids, n_group: int, topk_group: int, tol: float) -> bool:
    """Is ``ids`` a noaux_tc top-k of the biased scores ``b`` up to ``tol``? There must be a
    set of topk_group groups, each within tol of the topk_group-th best group score and
    holding every group that beats the best dropped group by more than tol, such that the
    chosen experts (distinct) lie in those groups and no other expert of them exceeds the
    smallest chosen score by more than tol. (A selection made exactly on scores within
    tol / 4 of ``b`` always passes: group scores move by at most twice that.)"""
    E = b.size
    G = E // n_group
    gs = np.sort(b.reshape(n_group, G), axis=1)[:, -2:].sum(1)
    desc = np.sort(gs)[::-1]
    cutoff = desc[topk_group - 1]
    chosen = [int(e) for e in ids]
    if len(set(chosen)) != len(chosen):
        return False
    chosen_set = set(chosen)
    low = min(b[e] for e in chosen)

    def below_chosen(g):
        return all(b[e] <= low + tol for e in range(g * G, (g + 1) * G) if e not in chosen_set)

    groups = {e // G for e in chosen}
    if any(gs[g] < cutoff - tol for g in groups):
        return False
    forced = ({g for g in range(n_group) if gs[g] > desc[topk_group] + tol}
              if topk_group < n_group else set(range(n_group)))
    kept = groups | forced
    if len(kept) > topk_group or not all(below_chosen(g) for g in kept):
        return False
    spare = [g for g in range(n_group) if g not in kept and gs[g] >= cutoff - tol and below_chosen(g)]
    return len(spare) >= topk_group - len(kept)


def check_routing(ref, got: dict, *, bias, n_group: int, topk_group: int, top_k: int,
                  n_experts: int) -> dict:
    """Compare routing; returns {'near_tie': [...], 'mismatch': [...]} and asserts the
    contract."""
    T = ref.ids.shape[0]
    gids = got["ids"].astype(np.int64)
    b = ref.scores + np.asarray(bias, np.float64)[None]
    near, diff = [], []
    for t in range(T):
        same = sorted(gids[t].tolist()) == sorted(ref.ids[t].tolist())
        if ref.margin[t] <= NEAR_TIE:
            near.append(t)
            kept = gids[t][gids[t] >= 0]
            assert kept.size > 0, t
            if kept.size == top_k:
                assert valid_selection(b[t], kept, n_group, topk_group, NEAR_TIE), t
            if not same:
                diff.append(t)
        else:
            assert same, (t, sorted(gids[t].tolist()), sorted(ref.ids[t].tolist()), ref.margin[t])
    # weights of the same expert
    for t in range(T):
        if t in diff:
            continue
        rw = {int(e): w for e, w in zip(ref.ids[t], ref.weights[t])}
        for e, w in zip(gids[t], got["weights"][t]):
            assert abs(w - rw[int(e)]) <= 1e-5 * abs(rw[int(e)]), (t, e, w, rw[int(e)])
    # entry lists: ascending tokens, slots consistent with the GPU's ids; the token sets
    # equal the oracle's except for near-tie tokens whose selection differs
    off, ent = got["offsets"], got["entries"]
    # slots dropped by the adaptive top-p carry id -1 and have no entry
    assert off[0] == 0 and off[-1] == int((gids >= 0).sum()) and np.all(np.diff(off) >= 0)
    dset = set(diff)
    for e in range(n_experts):
        g = ent[off[e]:off[e + 1]].astype(np.int64)
        toks, slots = g // top_k, g % top_k
        assert np.all(np.diff(toks) > 0), e
        assert np.all(gids[toks, slots] == e), e
        r = ref.entries[ref.offsets[e]:ref.offsets[e + 1]] // top_k
        gs_ = [t for t in toks.tolist() if t not in dset]
        rs_ = [t for t in r.tolist() if t not in dset]
        assert gs_ == rs_, e
    return {"near_tie": near, "mismatch": diff}


def out_errors(ref_out: np.ndarray, got: np.ndarray) -> tuple[float, float]:
    ref_out = np.asarray(ref_out, np.float64)
    got = np.asarray(got, np.float64)
    err = got - ref_out
    rel_l2 = float(np.linalg.norm(err) / max(np.linalg.norm(ref_out), 1e-300))
    max_rel = float(np.abs(err).max() / max(np.abs(ref_out).max(), 1e-300))
    return rel_l2, max_rel


def check_out(ref_out: np.ndarray, got: np.ndarray, rel_l2: float = REL_L2,
              max_rel: float = MAX_REL) -> tuple[float, float]:
    r, m = out_errors(ref_out, got)
    assert r <= rel_l2 and m <= max_rel, (r, m)
    return r, m
