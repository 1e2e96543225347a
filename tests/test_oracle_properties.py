"""Property-based pins of the oracle (no GPU): routing against brute force and the
layout against a direct re-sort, over random small shapes drawn by hypothesis, with
logits from a small set of values so that ties are common."""
import itertools

import numpy as np
import pytest
from hypothesis import given, settings
from hypothesis import strategies as st

import _oracles

TIE_VALUES = [-2.0, -0.0, 0.0, 0.5, 0.5, 1.0, 3.0]


@st.composite
def routing_case(draw):
    E = draw(st.integers(1, 9))
    k = draw(st.integers(1, E))
    T = draw(st.integers(1, 6))
    vals = draw(st.lists(st.sampled_from(TIE_VALUES), min_size=T * E, max_size=T * E))
    return np.array(vals, dtype=np.float32).reshape(T, E), k


def dominating_subset(row, k):
    """The one k-subset whose every member beats every left-out expert (larger
    logit, or an equal logit and a lower index)."""
    E = len(row)
    found = [set(S) for S in itertools.combinations(range(E), k)
             if all(row[i] > row[j] or (row[i] == row[j] and i < j)
                    for i in S for j in range(E) if j not in S)]
    assert len(found) == 1
    return found[0]


@pytest.mark.parametrize("impl", _oracles.NAMES)
@settings(max_examples=150, deadline=None)
@given(routing_case())
def test_route_matches_brute_force_with_ties(impl, case):
    O = _oracles.get(impl)
    logits, k = case
    ids, w = O.route(logits, k)
    for t in range(logits.shape[0]):
        row = logits[t].astype(np.float64)
        assert set(ids[t].tolist()) == dominating_subset(row, k)
        # listed in selection order: logit descending, index ascending
        keys = [(-row[e], e) for e in ids[t]]
        assert keys == sorted(keys)
        sel = row[ids[t]]
        np.testing.assert_allclose(w[t], np.exp(sel - sel.max()) / np.exp(sel - sel.max()).sum(), rtol=1e-12)


@st.composite
def layout_case(draw):
    R = draw(st.sampled_from([1, 2, 4]))
    E = R * draw(st.integers(1, 4))
    k = draw(st.integers(1, E))
    T = draw(st.integers(1, 20))
    ids = np.stack([np.array(draw(st.permutations(list(range(E)))))[:k] for _ in range(T)]).astype(np.int32)
    n_red = R * draw(st.integers(0, E // R))
    placement = draw(st.sampled_from(["linear", "round_robin"]))
    return ids, E, R, n_red, placement


@pytest.mark.parametrize("impl", _oracles.NAMES)
@settings(max_examples=150, deadline=None)
@given(layout_case())
def test_layout_is_the_stable_sort_by_physical_expert(impl, case):
    O = _oracles.get(impl)
    ids, E, R, n_red, placement = case
    T, k = ids.shape
    counts = np.bincount(ids.ravel(), minlength=E)
    emap = O.eplb_map(counts, R, n_red, placement)
    lay = O.dispatch_layout(ids, E, R, emap, placement)

    def phys(t, e):
        return int(emap["logical_to_phys"][e, t % emap["replica_count"][e]])

    order = sorted(((phys(t, int(ids[t, j])), t, j) for t in range(T) for j in range(k)), key=lambda a: a[:2])
    assert lay["row_to_token"].tolist() == [t for _, t, _ in order]
    for r, (_, t, j) in enumerate(order):
        assert lay["slot_to_row"][t, j] == r
    P = E + n_red
    assert lay["phys_counts"].sum() == T * k and lay["phys_offsets"][-1] == T * k
    assert np.array_equal(np.diff(lay["phys_offsets"]), lay["phys_counts"])
    # rank r owns physical ids r*P/R .. (r+1)*P/R - 1 and their rows
    per = P // R
    assert lay["rank_counts"].tolist() == [int(lay["phys_counts"][r * per:(r + 1) * per].sum()) for r in range(R)]
    # every replica carries its logical expert's tokens and nothing else
    for p in range(P):
        rows = range(int(lay["phys_offsets"][p]), int(lay["phys_offsets"][p + 1]))
        e = int(emap["phys_to_logical"][p])
        assert all(e in ids[lay["row_to_token"][r]] for r in rows)
    # the "before" statistics count each rank's base experts
    base_rank = [(e % R) if placement == "round_robin" else e // (E // R) for e in range(E)]
    before = [int(sum(counts[e] for e in range(E) if base_rank[e] == r)) for r in range(R)]
    assert lay["stats_before"]["max_rank"] == max(before)
