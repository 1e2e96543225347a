"""Pins for the CPU oracle: each test checks it against something other than itself
(brute force, library routines, closed forms, the pages' printed numbers)."""
import itertools
import json
import os
import random

import numpy as np
import pytest
import torch

import sys

import _oracles
import moe_inputs as mi
from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(params=_oracles.NAMES, autouse=True)
def oracle_impl(request, monkeypatch):
    """Every pin runs against both oracles: the numpy statement and the C++ one."""
    monkeypatch.setattr(sys.modules[__name__], "O", _oracles.get(request.param))
    return request.param


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ route
def brute_topk(l, k):
    """Enumerate every k-subset; keep the one that dominates all left-out experts
    (strictly larger logit, or equal logit and a lower index)."""
    E = len(l)
    winners = []
    for S in itertools.combinations(range(E), k):
        rest = [j for j in range(E) if j not in S]
        if all(l[i] > l[j] or (l[i] == l[j] and i < j) for i in S for j in rest):
            winners.append(set(S))
    assert len(winners) == 1
    return winners[0]


@pytest.mark.parametrize("E,k", [(1, 1), (4, 2), (6, 3), (8, 2), (8, 8), (10, 4)])
def test_route_brute_force_with_ties(E, k):
    rng = np.random.default_rng(E * 31 + k)
    for trial in range(40):
        # small integer-valued logits force many ties; signed zeros must tie too
        l = rng.integers(-2, 3, size=(1, E)).astype(np.float32)
        if trial % 3 == 0:
            l[0, rng.integers(0, E)] = -0.0
        ids, w = O.route(l, k)
        assert set(ids[0].tolist()) == brute_topk(l[0].tolist(), k)
        sel = l[0][ids[0]]
        # the chosen order: logit descending, then index ascending
        for a in range(k - 1):
            assert sel[a] > sel[a + 1] or (sel[a] == sel[a + 1] and ids[0][a] < ids[0][a + 1])
        assert abs(w.sum() - 1.0) < 1e-12


@pytest.mark.parametrize("E,k", [(8, 2), (10, 4), (12, 3)])
def test_route_selection_bias_brute_force(E, k):
    rng = np.random.default_rng(E + k)
    for trial in range(30):
        l = rng.integers(-3, 4, size=(1, E)).astype(np.float32)
        b = rng.integers(-2, 3, size=E).astype(np.float32)
        ids, w = O.route_selection_bias(l, b, k)
        score = (l[0] + b).tolist()
        assert set(ids[0].tolist()) == brute_topk(score, k)      # picked by logit + bias
        assert w.sum() == pytest.approx(1.0, abs=1e-15)
        lv = l[0][ids[0]].astype(np.float64)                      # weighted by the logits alone
        for a in range(k):
            for c in range(k):
                assert w[0, a] / w[0, c] == pytest.approx(np.exp(lv[a] - lv[c]), rel=1e-13)


def test_route_selection_bias_special_cases():
    rng = np.random.default_rng(3)
    l = rng.standard_normal((32, 16)).astype(np.float32)
    ids0, w0 = O.route(l, 4)
    ids1, w1 = O.route_selection_bias(l, np.zeros(16), 4)
    assert np.array_equal(ids0, ids1) and np.allclose(w0, w1, rtol=0, atol=1e-15)
    b = np.zeros(16, dtype=np.float32)
    b[5], b[9] = 1e4, -1e4              # always picked first / never picked
    ids, w = O.route_selection_bias(l, b, 4)
    assert (ids[:, 0] == 5).all() and not (ids == 9).any()
    # the bias moves picks only: a token whose unbiased top-4 holds expert 5 and not 9
    # keeps its experts and weights
    keep = [t for t in range(32) if 5 in ids0[t] and 9 not in ids0[t]]
    assert keep
    for t in keep:
        assert set(ids[t].tolist()) == set(ids0[t].tolist())
        assert np.allclose(np.sort(w[t]), np.sort(w0[t]), rtol=0, atol=1e-15)


def test_route_signed_zero_is_a_tie():
    l = np.array([[-0.0, 0.0, -1.0]], dtype=np.float32)
    ids, _ = O.route(l, 1)
    assert ids[0, 0] == 0


def test_route_k_equals_E_is_softmax():
    rng = np.random.default_rng(1)
    l = rng.standard_normal((16, 8)).astype(np.float32)
    ids, w = O.route(l, 8)
    ref = torch.softmax(torch.from_numpy(l).double(), dim=1).numpy()
    got = np.zeros_like(ref)
    np.put_along_axis(got, ids.astype(np.int64), w, axis=1)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-14)


def test_route_k1_is_argmax_weight_one():
    rng = np.random.default_rng(2)
    l = rng.standard_normal((64, 16)).astype(np.float32)
    ids, w = O.route(l, 1)
    assert np.array_equal(ids[:, 0], torch.argmax(torch.from_numpy(l), dim=1).numpy())
    assert np.all(w == 1.0)


def test_route_weights_two_forms_agree():
    l = mi.make_logits(mi.config("tiny_fp32"))
    _, w1 = O.route(l, 2)
    _, w2 = O.route_softmax_then_renorm(l, 2)
    np.testing.assert_allclose(w1, w2, rtol=0, atol=1e-12)


def test_route_rejects_non_finite():
    l = np.zeros((2, 4), dtype=np.float32)
    l[1, 2] = np.nan
    with pytest.raises(ValueError):
        O.route(l, 2)


# ------------------------------------------------------------------ layout
def brute_layout(ids, E, phys_of):
    T, k = ids.shape
    items = [(phys_of(t, int(ids[t, j])), t, j) for t in range(T) for j in range(k)]
    items_sorted = sorted(items, key=lambda a: (a[0], a[1]))
    row_to_token = [t for _, t, _ in items_sorted]
    slot_to_row = np.zeros((T, k), dtype=np.int64)
    for r, (_, t, j) in enumerate(items_sorted):
        slot_to_row[t, j] = r
    return row_to_token, slot_to_row


@pytest.mark.parametrize("T,E,k,R", [(1, 1, 1, 1), (3, 8, 2, 4), (64, 8, 2, 4), (257, 16, 4, 8)])
def test_layout_brute_force(T, E, k, R):
    l = np.random.default_rng(T + E).standard_normal((T, E)).astype(np.float32)
    ids, _ = O.route(l, k)
    lay = O.dispatch_layout(ids, E, R)
    r2t, s2r = brute_layout(ids, E, lambda t, e: e)
    assert lay["row_to_token"].tolist() == r2t
    assert np.array_equal(lay["slot_to_row"], s2r)
    cnt = [sum(1 for t in range(T) for j in range(k) if ids[t, j] == e) for e in range(E)]
    assert lay["phys_counts"].tolist() == cnt
    assert lay["phys_offsets"][-1] == T * k
    assert np.array_equal(np.diff(lay["phys_offsets"]), lay["phys_counts"])
    per = E // R
    assert lay["rank_counts"].tolist() == [sum(cnt[r * per:(r + 1) * per]) for r in range(R)]


def test_dispatch_figure_example():
    g = load("dispatch_figure.json")
    # 16 tokens (4 GPUs x 4), top-2 over 8 experts, 2 experts per GPU
    pairs = [(0, 1)] * 6 + [(6, 7)] * 2 + [(2, 4)] * 4 + [(3, 5)] * 4
    ids = np.array(pairs, dtype=np.int32)
    assert ids.shape == (g["gpus"] * g["tokens_per_gpu"], g["top_k"])
    lay = O.dispatch_layout(ids, g["experts"], g["ep"])
    assert lay["rank_counts"][0] == g["copies_gpu0"]
    assert lay["rank_counts"][3] == g["copies_gpu3"]
    st = lay["stats_after"]
    assert st["mean_rank"] == 8
    assert st["max_over_mean"] == pytest.approx(1.5)
    assert st["balancedness"] == pytest.approx(2 / 3)


def test_printed_ep256_column_from_printed_counts():
    """The section 5.2 table at EP 256 (one expert per card, no redundant slot), from
    its printed figures alone: with the hottest expert at 640 copies of 4096 x 8 picks
    over 256 experts (average 128), the contiguous placement and the rebalanced one
    both leave the busiest card at 640 / 128 = 5.00, whatever the other counts are.
    Any counts with that hottest value and total give the printed pair."""
    g = load("ep256_printed.json")
    total = g["tokens"] * g["top_k"]
    rng = np.random.default_rng(21)
    for _ in range(5):
        hot = int(rng.integers(0, g["experts"]))
        cold = [e for e in range(g["experts"]) if e != hot]
        rest = total - g["hottest"]
        # spread the remaining picks evenly, then move random amounts between cold
        # experts, keeping every count between 0 and the hottest
        counts = np.zeros(g["experts"], dtype=np.int64)
        counts[hot] = g["hottest"]
        counts[cold] = rest // len(cold)
        counts[cold[: rest % len(cold)]] += 1
        for _ in range(2000):
            a, b = rng.choice(cold, 2, replace=False)
            m = int(rng.integers(0, min(counts[a], g["hottest"] - counts[b]) + 1))
            counts[a] -= m
            counts[b] += m
        assert counts.max() == g["hottest"] and counts.sum() == total
        assert round(total / g["experts"]) == g["average"]
        st = O.rank_stats(O.linear_rank_counts(counts, g["ep"]), total)
        assert round(st["max_over_mean"], 2) == g["contiguous"]
        m = O.eplb_balanced_map(counts, g["ep"], 0)
        assert round(m["rank_load"].max() / m["rank_load"].mean(), 2) == g["rebalance"]


def test_balanced_map_worked_example():
    # Worked by hand from the page's steps: counts 10, 6, 3, 1 over 2 ranks with 2
    # redundant slots.  Slot 1 -> expert 0 (10 > 6), slot 2 -> expert 1 (6 > 5).
    # Replicas, heaviest first: e0 5, e0 5, e1 3, e1 3, e2 3, e3 1; S = 3 slots per
    # rank.  Ranks: e0 -> 0 (tie, lowest), e0 -> 1, e1 -> 0 (5 = 5), e1 -> 1,
    # e2 -> 0 (8 = 8), e3 -> 1 (rank 0 is full).  Loads 11 and 9.
    m = O.eplb_balanced_map(np.array([10, 6, 3, 1]), 2, 2)
    assert m["replica_count"].tolist() == [2, 2, 1, 1]
    assert m["phys_to_logical"].tolist() == [0, 1, 2, 0, 1, 3]
    assert m["phys_rank"].tolist() == [0, 0, 0, 1, 1, 1]
    assert m["logical_to_phys"].tolist() == [[0, 3, -1], [1, 4, -1], [2, -1, -1], [5, -1, -1]]
    assert m["rank_load"].tolist() == [11.0, 9.0]


def test_balanced_map_worked_example_one_hot_expert():
    # counts 100, 1, 1, 1 over 2 ranks with 2 redundant slots, worked by hand:
    # slot 1 -> e0 (100 > 1), slot 2 -> e0 again (50 > 1): e0 has 3 replicas of 100/3.
    # S = 3.  Replicas: e0 r0 -> rank 0 (tie, lowest); e0 r1 -> rank 1 (0 < 33.3);
    # e0 r2 -> rank 0 (tie at 33.3, lowest); e1 -> rank 1 (33.3 < 66.7); e2 -> rank 1
    # (34.3 < 66.7), which fills it; e3 -> rank 0.
    m = O.eplb_balanced_map(np.array([100, 1, 1, 1]), 2, 2)
    third = 100 / 3
    assert m["replica_count"].tolist() == [3, 1, 1, 1]
    assert m["phys_rank"].tolist() == [0, 0, 0, 1, 1, 1]
    assert m["phys_to_logical"].tolist() == [0, 0, 3, 0, 1, 2]
    assert m["logical_to_phys"].tolist() == [[0, 3, 1], [4, -1, -1], [5, -1, -1], [2, -1, -1]]
    assert m["rank_load"].tolist() == [third + third + 1.0, third + 1.0 + 1.0]


def test_balanced_map_equal_counts_deal_round_robin():
    # all loads equal: replicas arrive in expert order and every card is the lightest
    # in turn, so expert e lands on card e mod R (slot e div R)
    E, R = 12, 4
    m = O.eplb_balanced_map(np.full(E, 5), R, 0)
    S = E // R
    for e in range(E):
        p = m["logical_to_phys"][e, 0]
        assert m["phys_rank"][p] == e % R and p == (e % R) * S + e // R
    assert m["rank_load"].tolist() == [15.0] * R


def test_balanced_map_invariants():
    rng = np.random.default_rng(11)
    for E, R, n_red in ((256, 32, 32), (64, 8, 40), (30, 4, 10)):
        counts = rng.integers(0, 1000, size=E)
        counts[3] = 40000
        m = O.eplb_balanced_map(counts, R, n_red)
        P, S = E + n_red, (E + n_red) // R
        assert np.bincount(m["phys_rank"], minlength=R).tolist() == [S] * R
        assert m["replica_count"].sum() == P and m["replica_count"].min() >= 1
        seen = np.zeros(P, dtype=bool)
        for e in range(E):
            row = m["logical_to_phys"][e]
            n = m["replica_count"][e]
            assert (row[n:] == -1).all() and (row[:n] >= 0).all()
            assert (m["phys_to_logical"][row[:n]] == e).all() and not seen[row[:n]].any()
            seen[row[:n]] = True
            assert (row[:n] // S == m["phys_rank"][row[:n]]).all()
        assert seen.all()
        # the rank loads are the per-replica loads summed over each rank's slots
        per = counts / m["replica_count"]
        again = np.zeros(R)
        np.add.at(again, m["phys_rank"], per[m["phys_to_logical"]])
        assert np.allclose(again, m["rank_load"], rtol=1e-12, atol=0)
        # the hottest expert (40000) holds the most replicas
        assert m["replica_count"][3] == m["replica_count"].max()


def test_eplb_window_sum_by_hand():
    steps = [[1, 2], [3, 4], [5, 6], [7, 8]]
    assert O.eplb_window_sum(steps[:1], 3).tolist() == [1, 2]            # fewer steps than W
    assert O.eplb_window_sum(steps[:3], 3).tolist() == [9, 12]
    assert O.eplb_window_sum(steps, 3).tolist() == [15, 18]              # the oldest step left
    assert O.eplb_window_sum(steps, 1).tolist() == [7, 8]


# ------------------------------------------------------------------ EPLB
def test_eplb_map_geometry_and_hot_list():
    rng = np.random.default_rng(5)
    counts = rng.integers(0, 50, size=256)
    counts[17] = counts[200] = 1000          # a tie at the top: lower index first
    m = O.eplb_map(counts, 32, 32)
    g = load("expert_arithmetic.json")
    assert m["P"] // 32 == g["physical_per_rank_256_32_32"]
    assert np.bincount(m["phys_rank"], minlength=32).tolist() == [9] * 32
    hot = m["hot"].tolist()
    assert hot[0] == 17 and hot[1] == 200
    # brute force: every hot expert beats every cold one on (count desc, index asc)
    cold = [e for e in range(256) if e not in hot]
    for h in hot:
        for c in cold:
            assert counts[h] > counts[c] or (counts[h] == counts[c] and h < c)
    # primaries are the linear blocks; replica j on rank j mod 32
    for e in range(256):
        p = m["logical_to_phys"][e, 0]
        assert m["phys_rank"][p] == e // 8 and m["phys_to_logical"][p] == e
    for j, e in enumerate(hot):
        p = m["logical_to_phys"][e, 1]
        assert m["phys_rank"][p] == j % 32 and m["phys_to_logical"][p] == e
    assert sorted(m["replica_count"].tolist()).count(2) == 32
    assert O.eplb_map(counts[:256], 8, 8)["P"] // 8 == g["physical_per_rank_256_8_8"]


def test_eplb_token_split_by_parity():
    cfg = mi.config("prefill_bf16_skew_eplb").scaled(T=512)
    l = mi.make_logits(cfg)
    ids, _ = O.route(l, cfg.k)
    m = O.eplb_map(np.bincount(ids.ravel(), minlength=cfg.E), cfg.R, cfg.n_redundant)
    lay = O.dispatch_layout(ids, cfg.E, cfg.R, m)
    for e in m["hot"][:8]:
        even = sum(1 for t in range(cfg.T) if e in ids[t] and t % 2 == 0)
        odd = sum(1 for t in range(cfg.T) if e in ids[t] and t % 2 == 1)
        assert lay["phys_counts"][m["logical_to_phys"][e, 0]] == even
        assert lay["phys_counts"][m["logical_to_phys"][e, 1]] == odd
    r2t, s2r = brute_layout(ids, cfg.E, lambda t, e: int(m["logical_to_phys"][e, t % m["replica_count"][e]]))
    assert lay["row_to_token"].tolist() == r2t
    assert np.array_equal(lay["slot_to_row"], s2r)


def test_round_robin_placement_by_hand():
    """8 experts on 4 ranks, one copy per token: round-robin deals experts 0..7 to
    ranks 0,1,2,3,0,1,2,3; the busiest rank is worked out by hand."""
    counts = [10, 0, 3, 5, 2, 7, 1, 4]
    ids = np.repeat(np.arange(8), counts).astype(np.int32)[:, None]
    lay = O.dispatch_layout(ids, 8, 4, O.eplb_map(np.zeros(8), 4, 0, "round_robin"), "round_robin")
    # rank 0: e0 + e4 = 12; rank 1: e1 + e5 = 7; rank 2: e2 + e6 = 4; rank 3: e3 + e7 = 9
    assert lay["rank_counts"].tolist() == [12, 7, 4, 9]
    assert lay["stats_before"]["max_rank"] == 12 and lay["stats_after"]["max_rank"] == 12
    assert lay["stats_before"]["max_over_mean"] == 1.5
    # the linear placement of the same counts: 10, 8, 9, 5
    lin = O.dispatch_layout(ids, 8, 4)
    assert lin["rank_counts"].tolist() == [10, 8, 9, 5] and lin["stats_before"]["max_over_mean"] == 1.25


@pytest.mark.parametrize("E,R,n_red", [(256, 32, 0), (256, 32, 32), (64, 8, 16), (12, 3, 6)])
def test_round_robin_map_geometry(E, R, n_red):
    rng = np.random.default_rng(E + n_red)
    counts = rng.integers(0, 40, size=E)
    m = O.eplb_map(counts, R, n_red, "round_robin")
    lin = O.eplb_map(counts, R, n_red)
    S = (E + n_red) // R
    for e in range(E):
        p = m["logical_to_phys"][e, 0]
        assert p == (e % R) * S + e // R                  # rank e mod R, local slot e div R
        assert m["phys_rank"][p] == e % R and m["phys_to_logical"][p] == e
    assert np.bincount(m["phys_rank"], minlength=R).tolist() == [S] * R
    assert sorted(m["phys_to_logical"][m["phys_rank"] == 0].tolist()[:E // R]) == list(range(0, E, R))
    # replicas do not depend on the base placement
    assert np.array_equal(m["hot"], lin["hot"])
    for e in m["hot"]:
        assert m["logical_to_phys"][e, 1] == lin["logical_to_phys"][e, 1]
    assert np.array_equal(m["replica_count"], lin["replica_count"])


@pytest.mark.parametrize("E,R", [(8, 1), (8, 8), (256, 256)])
def test_round_robin_equals_linear_when_degenerate(E, R):
    """One rank, or one expert per rank: both strategies give every rank the same experts."""
    counts = np.arange(E)[::-1]
    a, b = O.eplb_map(counts, R, 0, "round_robin"), O.eplb_map(counts, R, 0)
    for key in ("phys_to_logical", "phys_rank", "logical_to_phys"):
        assert np.array_equal(a[key], b[key])


@pytest.mark.parametrize("T,E,k,R", [(3, 8, 2, 4), (200, 16, 4, 8), (257, 32, 8, 4)])
def test_round_robin_layout_brute_force(T, E, k, R):
    """Rows in order (rank e mod R, slot e div R, token), straight from the rule."""
    l = np.random.default_rng(T * E).standard_normal((T, E)).astype(np.float32)
    ids, _ = O.route(l, k)
    lay = O.dispatch_layout(ids, E, R, O.eplb_map(np.zeros(E), R, 0, "round_robin"), "round_robin")
    r2t, s2r = brute_layout(ids, E, lambda t, e: (e % R) * (E // R) + e // R)
    assert lay["row_to_token"].tolist() == r2t
    assert np.array_equal(lay["slot_to_row"], s2r)
    per_rank = [sum(1 for t in range(T) for j in range(k) if ids[t, j] % R == r) for r in range(R)]
    assert lay["rank_counts"].tolist() == per_rank
    assert lay["stats_before"]["max_rank"] == max(per_rank)


def test_round_robin_layer_output_equals_linear():
    """The placement moves rows between ranks; the layer's result is unchanged."""
    cfg = mi.config("tiny_fp32")
    l = mi.make_logits(cfg)
    x = np.random.default_rng(3).standard_normal((cfg.T, cfg.d)).astype(np.float32)
    wt = tiny_weights(cfg, 4)
    a = O.layer_forward(cfg, l, x, wt)
    b = O.layer_forward(cfg.scaled(expert_placement=1), l, x, wt)
    assert np.array_equal(a["out"], b["out"])
    assert not np.array_equal(a["layout"]["row_to_token"], b["layout"]["row_to_token"])


# ------------------------------------------------------------------ number formats
def test_bf16_rounding_matches_torch():
    v = np.random.default_rng(3).standard_normal(100000) * 10.0
    ref = torch.from_numpy(v).float().bfloat16().double().numpy()
    assert np.array_equal(O.round_bf16(v), ref)


def test_e4m3_table_landmarks():
    assert O.e4m3_value(0x7E) == 448.0
    assert O.e4m3_value(0x08) == 2.0 ** -6
    assert O.e4m3_value(0x01) == 2.0 ** -9
    assert np.isnan(O.e4m3_value(0x7F))
    assert O.e4m3_encode(np.array([1000.0, -1e9, 448.0], np.float32)).tolist() == [0x7E, 0xFE, 0x7E]


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(4)
    v = np.concatenate([
        rng.standard_normal(200000) * 50,
        rng.standard_normal(50000) * 0.01,                      # subnormal range
        np.array([O.e4m3_value(c) for c in range(127)]),        # exact values
        (np.array([O.e4m3_value(c) for c in range(126)]) + np.array([O.e4m3_value(c) for c in range(1, 127)])) / 2,  # ties
    ]).astype(np.float32)
    v = v[np.abs(v) <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(v), ref)


def test_quantize_groups_bound_and_amax():
    rng = np.random.default_rng(6)
    v = (rng.standard_normal((32, 512)) * rng.uniform(0.01, 100, size=(32, 1))).astype(np.float32)
    v[3, :128] = 0.0
    q, s = O.quantize_groups(v)
    deq = O.dequantize_groups(q, s)
    assert s[3, 0] == 1.0 and np.all(q[3, :128] == 0)
    # e4m3 keeps 3 mantissa bits: half-ulp relative bound 2^-4 for normals,
    # absolute bound scale * 2^-10 in the subnormal range
    bound = np.maximum(np.abs(v) * 2.0 ** -4, np.repeat(s, 128, axis=1) * 2.0 ** -10)
    assert np.all(np.abs(deq - v) <= bound * (1 + 1e-6))
    g = np.abs(v.reshape(32, 4, 128)).max(axis=2)
    assert np.all((g == 0) | (np.abs(q.reshape(32, 4, 128)) .max(axis=2) > 0))
    assert np.all(np.isin((q.reshape(32, 4, 128) & 0x7F).max(axis=2)[g > 0], [0x7E]))


def test_dequantize_groups_bf16_matches_torch():
    """FP8 dispatch, receive side: torch's e4m3 decode, a float32 multiply and its
    bf16 conversion give the same values."""
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 256, size=(24, 384)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x7E                          # no NaN codes
    codes[0, :256] = np.arange(256, dtype=np.uint8)
    codes[0, :256][(codes[0, :256] & 0x7F) == 0x7F] = 0
    scales = (2.0 ** rng.uniform(-12, 12, size=(24, 3))).astype(np.float32)
    got = O.dequantize_groups_bf16(codes, scales)
    tv = torch.from_numpy(codes).view(torch.float8_e4m3fn).float()
    ts = torch.from_numpy(np.repeat(scales, 128, axis=1))
    ref = (tv * ts).bfloat16().double().numpy()
    assert np.array_equal(got, ref)


def test_fp8_dispatch_lossless_on_the_e4m3_grid():
    """Tokens whose 128-channel groups hold e4m3 values times 2^-4 with amax 28 have
    scale 2^-4 exactly, so the e4m3 dispatch returns them unchanged and the layer's
    output equals the plain bf16 dispatch's."""
    cfg = mi.config("prefill_bf16_skew").scaled(T=24, d=256, E=4, k=2, I=128, R=2, shared=False, zipf_bias=False)
    rng = np.random.default_rng(12)
    grid = O.e4m3_decode(np.arange(0x7F, dtype=np.uint8))            # finite non-negative values
    x = (rng.choice(grid, size=(cfg.T, cfg.d)) * rng.choice([-1.0, 1.0], size=(cfg.T, cfg.d)) / 16.0)
    x[:, ::128] = 448.0 / 16.0                                       # every group's amax is 28
    x = x.astype(np.float32)
    l = rng.standard_normal((cfg.T, cfg.E)).astype(np.float32)
    wt = tiny_weights(cfg, 13)
    a = O.layer_forward(cfg, l, x, wt)
    b = O.layer_forward(cfg.scaled(fp8_dispatch=1), l, x, wt)
    assert np.all(b["x_scales"] == np.float32(1 / 16))
    assert np.array_equal(a["out"], b["out"])
    # off the grid the dispatch rounds: the rows move by at most e4m3's half ulp and
    # bf16's, and the output changes
    x2 = rng.standard_normal((cfg.T, cfg.d)).astype(np.float32)
    a2 = O.layer_forward(cfg, l, x2, wt)
    b2 = O.layer_forward(cfg.scaled(fp8_dispatch=1), l, x2, wt)
    deq = O.dequantize_groups_bf16(b2["x_q"], b2["x_scales"])
    sc = np.repeat(b2["x_scales"], 128, axis=1)
    bound = (np.abs(x2) * 2.0 ** -4 + sc * 2.0 ** -10) * (1 + 2.0 ** -8) + np.abs(x2) * 2.0 ** -8
    assert np.all(np.abs(deq - x2) <= bound)
    assert not np.array_equal(a2["out"], b2["out"])
    # the shared expert is not dispatched: its contribution does not change
    cs = cfg.scaled(shared=True, E=1, k=1, R=1)
    l1 = np.zeros((cfg.T, 1), np.float32)
    a3 = O.layer_forward(cs, l1, x2, wt, eplb_enabled=False)
    b3 = O.layer_forward(cs.scaled(fp8_dispatch=1), l1, x2, wt, eplb_enabled=False)
    sh = O.swiglu_expert(x2.astype(np.float64), wt("ws_gate", 0).astype(np.float64),
                         wt("ws_up", 0).astype(np.float64), wt("ws_down", 0).astype(np.float64), "bf16")
    w64 = [wt(n, 0).astype(np.float64) for n in ("w_gate", "w_up", "w_down")]
    deq = O.dequantize_groups_bf16(b3["x_q"], b3["x_scales"])
    # one expert at weight 1: out = routed FFN of the dispatched rows + shared FFN of x
    assert np.allclose(a3["out"], O.swiglu_expert(x2.astype(np.float64), *w64, "bf16") + sh, rtol=0, atol=1e-12)
    assert np.allclose(b3["out"], O.swiglu_expert(deq, *w64, "bf16") + sh, rtol=0, atol=1e-12)


def test_layer_selection_bias_special_cases():
    cfg = mi.config("tiny_fp32")
    l = mi.make_logits(cfg)
    x = np.random.default_rng(14).standard_normal((cfg.T, cfg.d)).astype(np.float32)
    wt = tiny_weights(cfg, 15)
    plain = O.layer_forward(cfg, l, x, wt)
    zero = O.layer_forward(cfg, l, x, wt, selection_bias=np.zeros(cfg.E, np.float32))
    assert np.array_equal(plain["out"], zero["out"])
    # a bias far below every logit keeps expert 3 out of every selection
    b = np.zeros(cfg.E, np.float32)
    b[3] = -1e4
    res = O.layer_forward(cfg, l, x, wt, selection_bias=b)
    assert res["layout"]["logical_counts"][3] == 0 and 3 not in res["topk_ids"]


def test_quantize_blocks_matches_groups_on_blocks():
    rng = np.random.default_rng(7)
    w = rng.standard_normal((256, 384)).astype(np.float32)
    q, s = O.quantize_blocks(w)
    assert s.shape == (2, 3)
    for bi in range(2):
        for bj in range(3):
            blk = w[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
            assert s[bi, bj] == np.float32(np.abs(blk).max()) / np.float32(448)
            ref = torch.from_numpy(blk / s[bi, bj]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(q[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128], ref)


# ------------------------------------------------------------------ FFN and combine
def torch_swiglu(x, wg, wu, wd):
    x, wg, wu, wd = (torch.from_numpy(np.asarray(a, dtype=np.float64)) for a in (x, wg, wu, wd))
    return (torch.nn.functional.silu(x @ wg) * (x @ wu)) @ wd


def tiny_weights(cfg, seed):
    rng = np.random.default_rng(seed)
    W = {}
    for e in range(cfg.E):
        W[("w_gate", e)] = (rng.standard_normal((cfg.d, cfg.I)) / np.sqrt(cfg.d)).astype(np.float32)
        W[("w_up", e)] = (rng.standard_normal((cfg.d, cfg.I)) / np.sqrt(cfg.d)).astype(np.float32)
        W[("w_down", e)] = (rng.standard_normal((cfg.I, cfg.d)) / np.sqrt(cfg.I)).astype(np.float32)
    for n in ("gate", "up", "down"):
        W[("ws_" + n, 0)] = W[("w_" + n, 0)] * np.float32(0.5)
    return lambda which, e: W[(which, e)]


def test_ffn_single_expert_is_dense_swiglu():
    cfg = mi.config("tiny_fp32").scaled(E=1, k=1, R=1)
    x = np.random.default_rng(8).standard_normal((cfg.T, cfg.d)).astype(np.float32)
    wt = tiny_weights(cfg, 9)
    res = O.layer_forward(cfg, np.zeros((cfg.T, 1), np.float32), x, wt)
    ref = torch_swiglu(x, wt("w_gate", 0), wt("w_up", 0), wt("w_down", 0)).numpy()
    np.testing.assert_allclose(res["out"], ref, rtol=1e-12, atol=1e-12)


def test_ffn_top1_uses_argmax_expert():
    cfg = mi.config("tiny_fp32").scaled(k=1)
    rng = np.random.default_rng(10)
    x = rng.standard_normal((cfg.T, cfg.d)).astype(np.float32)
    l = rng.standard_normal((cfg.T, cfg.E)).astype(np.float32)
    wt = tiny_weights(cfg, 11)
    res = O.layer_forward(cfg, l, x, wt)
    am = torch.argmax(torch.from_numpy(l), dim=1).numpy()
    for t in range(cfg.T):
        e = am[t]
        ref = torch_swiglu(x[t:t + 1], wt("w_gate", e), wt("w_up", e), wt("w_down", e)).numpy()[0]
        np.testing.assert_allclose(res["out"][t], ref, rtol=1e-12, atol=1e-12)


def test_ffn_all_experts_softmax_mixture_with_shared():
    cfg = mi.config("tiny_fp32").scaled(k=8, shared=True, T=8)
    rng = np.random.default_rng(12)
    x = rng.standard_normal((cfg.T, cfg.d)).astype(np.float32)
    l = rng.standard_normal((cfg.T, cfg.E)).astype(np.float32)
    wt = tiny_weights(cfg, 13)
    res = O.layer_forward(cfg, l, x, wt)
    p = torch.softmax(torch.from_numpy(l).double(), dim=1)
    ref = torch_swiglu(x, wt("ws_gate", 0), wt("ws_up", 0), wt("ws_down", 0))
    for e in range(cfg.E):
        ref = ref + p[:, e:e + 1] * torch_swiglu(x, wt("w_gate", e), wt("w_up", e), wt("w_down", e))
    np.testing.assert_allclose(res["out"], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_identity_experts_return_x():
    cfg = mi.config("tiny_fp32")
    x = mi.make_x(cfg).astype(np.float64)
    ids, w = O.route(mi.make_logits(cfg), cfg.k)
    lay = O.dispatch_layout(ids, cfg.E, cfg.R)
    xp = O.permute(x, lay["row_to_token"])
    np.testing.assert_allclose(O.combine(xp, lay["slot_to_row"], w), x, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(O.combine(xp, lay["slot_to_row"], w, shared=x), 2 * x, rtol=1e-14, atol=1e-14)


def test_dispatch_bytes_and_expert_size_arithmetic():
    g = load("expert_arithmetic.json")
    cfg = mi.config("decode_bf16")
    assert 3 * cfg.d * cfg.I == g["expert_params_glm"]
    assert round(3 * cfg.d * cfg.I / 1e6, 1) == g["expert_mb_fp8_glm"]   # one byte per e4m3 weight
    T = 4
    x = np.zeros((T, cfg.d), dtype=np.uint16)                           # bf16 rows
    ids = np.stack([np.arange(cfg.k)] * T).astype(np.int32)
    lay = O.dispatch_layout(ids, cfg.E, cfg.R)
    assert O.permute(x, lay["row_to_token"]).nbytes // T == g["a2a_bytes_per_token_glm"]
    assert round(3 * 7168 * 2048 / 1e6) == g["expert_params_dsv3_approx_m"]
    assert round(8 * 7168 * 1 / 1000) == g["dispatch_fp8_bytes_dsv3_approx_kb"]
    assert round(8 * 7168 * 2 / 1000) == g["combine_bf16_bytes_dsv3_approx_kb"]


# ------------------------------------------------------------------ rounding points of the expert FFN
# One token, d = 1, x = [1]: with every gate weight 64, g = 64 and silu(64) = 64
# exactly in float64 (e^-64 < 2^-53, so 1 + e^-64 rounds to 1); h = 64 * u is then
# set by the up weights alone, and y = h . w_down by the down weights.  Every value
# below is a dyadic rational worked out by hand.
def one_token_expert(u, wd):
    u = np.asarray(u, dtype=np.float64)[None, :]
    I = u.shape[1]
    wd = np.asarray(wd, dtype=np.float64).reshape(I, 1)
    return np.ones((1, 1)), np.full((1, I), 64.0), u, wd


def test_bf16_mode_rounds_h_at_a_tie():
    # h = 64 (2^-6 + 2^-14) = 1 + 2^-8, halfway between the bf16 values 1 and 1 + 2^-7:
    # round-to-nearest-even keeps 1.  y = 3 h: 3 with h rounded; unrounded,
    # 3 + 3 * 2^-8 lies 3/4 of the way to the next bf16 value 3 + 2^-6.
    x, wg, wu, wd = one_token_expert([2.0 ** -6 + 2.0 ** -14], [3.0])
    assert O.swiglu_expert(x, wg, wu, wd, "bf16")[0, 0] == 3.0
    assert O.swiglu_expert(x, wg, wu, wd, "fp32")[0, 0] == 3.0 + 3.0 * 2.0 ** -8


def test_bf16_mode_rounds_y():
    # h = 1 exactly; y = 1 + 2^-8 is a bf16 tie and rounds to 1; the fp32 mode keeps it
    x, wg, wu, wd = one_token_expert([2.0 ** -6], [1.0 + 2.0 ** -8])
    assert O.swiglu_expert(x, wg, wu, wd, "bf16")[0, 0] == 1.0
    assert O.swiglu_expert(x, wg, wu, wd, "fp32")[0, 0] == 1.0 + 2.0 ** -8
    # y = 1 + 3 * 2^-8 is a tie between 1 + 2^-7 and 1 + 2^-6: the even one is 1 + 2^-6
    x, wg, wu, wd = one_token_expert([2.0 ** -6], [1.0 + 3.0 * 2.0 ** -8])
    assert O.swiglu_expert(x, wg, wu, wd, "bf16")[0, 0] == 1.0 + 2.0 ** -6


def test_bf16_mode_equals_fp32_mode_on_bf16_exact_values():
    # h = 1.5, 0.25, -2 (bf16-exact) and y = 1.5 * 2 + 0.25 * 4 - 2 * 0.5 = 3: no rounding bites
    x, wg, wu, wd = one_token_expert([1.5 / 64, 0.25 / 64, -2.0 / 64], [2.0, 4.0, 0.5])
    a = O.swiglu_expert(x, wg, wu, wd, "bf16")
    b = O.swiglu_expert(x, wg, wu, wd, "fp32")
    assert a[0, 0] == b[0, 0] == 3.0


def fp8_two_group_row():
    # I = 256: group 0 (channels 0-127) holds h = 448 at channel 0, so its scale is 1;
    # group 1 (channels 128-255) holds 28 at channel 128, so its scale is 28/448 = 2^-4,
    # and h = 3 * 2^-10 at channel 129.  Per 128 channels, 3 * 2^-10 / 2^-4 = 3 * 2^-6
    # = 1.5 * 2^-5 is an e4m3 normal (mantissa 0.5), so it comes back exactly.  One scale
    # for all 256 channels (448 / 448 = 1) puts it at 1.5 * 2^-9, halfway between the
    # subnormals 2^-9 and 2^-8, where the even code gives 2^-8.
    # Channel 1 holds 1 + 2^-5, which scale 1 rounds to the e4m3 value 1.
    u = np.zeros(256)
    u[0], u[128], u[129], u[1] = 448.0 / 64, 28.0 / 64, 3.0 * 2.0 ** -10 / 64, (1.0 + 2.0 ** -5) / 64
    return u


def test_fp8_mode_quantises_h_per_128_channels():
    u = fp8_two_group_row()
    wd = np.zeros(256)
    wd[129] = 1.0
    x, wg, wu, wdm = one_token_expert(u, wd)
    assert O.swiglu_expert(x, wg, wu, wdm, "fp8")[0, 0] == 3.0 * 2.0 ** -10
    wd = np.zeros(256)
    wd[1] = 1.0
    x, wg, wu, wdm = one_token_expert(u, wd)
    assert O.swiglu_expert(x, wg, wu, wdm, "fp8")[0, 0] == 1.0
    assert O.swiglu_expert(x, wg, wu, wdm, "fp32")[0, 0] == 1.0 + 2.0 ** -5


def test_fp8_mode_rounds_y_to_bf16():
    # h = 448 and 0: codes exact with scale 1; y = 448 * (1 + 2^-8) / 448 ... take
    # w_down = (1 + 2^-8) / 448 at channel 0: y = 1 + 2^-8, the bf16 tie that rounds to 1
    u = np.zeros(128)
    u[0] = 448.0 / 64
    wd = np.zeros(128)
    wd[0] = 2.0 ** -6 * (1.0 + 2.0 ** -8) / 7.0          # 448 = 7 * 2^6
    x, wg, wu, wdm = one_token_expert(u, wd)
    y32 = O.swiglu_expert(x, wg, wu, wdm, "fp32")[0, 0]
    assert abs(y32 - (1.0 + 2.0 ** -8)) < 1e-15
    assert O.swiglu_expert(x, wg, wu, wdm, "fp8")[0, 0] == 1.0


# ------------------------------------------------------------------ the bf16 rounding envelope
def test_bf16_bracket_by_hand():
    lo, hi = O.bf16_bracket(np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 2.0 ** -9, -3.0 - 2.0 ** -7, 0.0, 1e-45, -2.0]))
    # bf16-exact values bracket themselves; 1 + 2^-8 (a tie) and 1 + 2^-9 sit between
    # 1 and 1 + 2^-7; -3 - 2^-7 between -3 - 2^-6 and -3; 1e-45 between 0 and 2^-133
    assert lo.tolist() == [1.0, 1.0, 1.0, -3.0 - 2.0 ** -6, 0.0, 0.0, -2.0]
    assert hi.tolist() == [1.0, 1.0 + 2.0 ** -7, 1.0 + 2.0 ** -7, -3.0, 0.0, 2.0 ** -133, -2.0]


def test_layer_envelope_holds_the_round_to_nearest_output():
    for cfg in (mi.config("prefill_bf16_skew").scaled(T=40, d=128, E=8, I=128, R=4), mi.config("tiny_fp32"),
                mi.config("prefill_fp8_skew").scaled(T=40, d=128, E=8, I=128, R=4)):
        x = mi.make_x(cfg)
        l = mi.make_logits(cfg)
        wt = tiny_weights(cfg, 17)
        res = O.layer_forward(cfg, l, x, wt)
        assert np.all(res["out_lo"] <= res["out"] + 1e-12) and np.all(res["out"] <= res["out_hi"] + 1e-12)
        if cfg.dtype == "fp32":            # nothing is rounded: the envelope is the output
            assert np.allclose(res["out_lo"], res["out"], rtol=0, atol=1e-15)
            assert np.allclose(res["out_hi"], res["out"], rtol=0, atol=1e-15)
        else:                              # at most one bf16 step of each y, weighted
            assert np.all(res["out_hi"] - res["out_lo"] <= 2.0 ** -7 * (np.abs(res["out"]) + 4.0))
            assert np.any(res["out_hi"] > res["out_lo"])


def test_layer_envelope_by_hand():
    # one token, E = k = 1 with weight 1, d = 1: y = h w_down = 1 + 2^-8 exactly (the
    # bf16 tie), so the envelope is [1, 1 + 2^-7] and the rounded output 1
    cfg = mi.config("prefill_bf16_skew").scaled(T=1, d=128, E=1, k=1, I=128, R=1, shared=False, zipf_bias=False)
    wg = np.zeros((128, 128), np.float32)
    wu = np.zeros((128, 128), np.float32)
    wd = np.zeros((128, 128), np.float32)
    wg[0, 0], wu[0, 0] = 64.0, 2.0 ** -6            # h_0 = silu(64) * 1 = 64 * 2^-6 = 1
    wd[0, 0] = 1.0 + 2.0 ** -8                       # y_0 = 1 + 2^-8
    W = {"w_gate": wg, "w_up": wu, "w_down": wd}
    x = np.zeros((1, 128), np.float32)
    x[0, 0] = 1.0
    res = O.layer_forward(cfg, np.zeros((1, 1), np.float32), x, lambda which, e: W[which])
    assert res["out"][0, 0] == 1.0
    assert res["out_lo"][0, 0] == 1.0 and res["out_hi"][0, 0] == 1.0 + 2.0 ** -7


# ------------------------------------------------------------------ planted mistakes
def test_pins_catch_planted_mistakes(monkeypatch, oracle_impl):
    """Plant plausible slips in the numpy oracle and check that a pin above fails
    (the C++ oracle's planted slips are compiled variants: test_oracle_cpp.py)."""
    if oracle_impl != "numpy":
        pytest.skip("monkeypatched slips are for the numpy oracle")
    cfg = mi.config("tiny_fp32").scaled(E=1, k=1, R=1)
    x = np.random.default_rng(8).standard_normal((cfg.T, cfg.d)).astype(np.float32)
    wt = tiny_weights(cfg, 9)
    ref = torch_swiglu(x, wt("w_gate", 0), wt("w_up", 0), wt("w_down", 0)).numpy()
    real = O.swiglu_expert_exact

    def swapped(x64, wg, wu, wd, mode):           # gate and up exchanged
        return real(x64, wu, wg, wd, mode)

    monkeypatch.setattr(O, "swiglu_expert_exact", swapped)
    out = O.layer_forward(cfg, np.zeros((cfg.T, 1), np.float32), x, wt)["out"]
    assert not np.allclose(out, ref, rtol=1e-6, atol=1e-6)
    monkeypatch.setattr(O, "swiglu_expert_exact", real)

    monkeypatch.setattr(O, "silu", lambda z: z / (1.0 + np.exp(z)))   # sign slip
    out = O.layer_forward(cfg, np.zeros((cfg.T, 1), np.float32), x, wt)["out"]
    assert not np.allclose(out, ref, rtol=1e-6, atol=1e-6)
    monkeypatch.undo()

    # a tie-break slip (equal logits -> higher index) disagrees with the brute force
    l = np.array([[1.0, 2.0, 2.0, 0.0]], dtype=np.float32)
    ids_bad = 3 - np.argsort(-l[:, ::-1], axis=1, kind="stable")[:, :1]
    assert set(ids_bad[0].tolist()) != brute_topk(l[0].tolist(), 1)
    assert set(O.route(l, 1)[0][0].tolist()) == brute_topk(l[0].tolist(), 1)

    # a round-robin map that keeps the linear slots fails the hand-worked rank loads
    ids = np.repeat(np.arange(8), [10, 0, 3, 5, 2, 7, 1, 4]).astype(np.int32)[:, None]
    lay = O.dispatch_layout(ids, 8, 4, O.eplb_map(np.zeros(8), 4, 0, "linear"), "round_robin")
    assert lay["rank_counts"].tolist() != [12, 7, 4, 9]

    # the rounding points of the expert FFN: h left unrounded, h quantised over all
    # 256 channels at once, y left unrounded
    def check_rounding_pins():
        for pin in (test_bf16_mode_rounds_h_at_a_tie, test_bf16_mode_rounds_y,
                    test_fp8_mode_quantises_h_per_128_channels, test_fp8_mode_rounds_y_to_bf16):
            try:
                pin()
            except AssertionError:
                return False
        return True

    assert check_rounding_pins()
    real_h, real_y = O.stored_h, O.stored_y
    monkeypatch.setattr(O, "stored_h", lambda h, mode: h if mode == "bf16" else real_h(h, mode))
    assert not check_rounding_pins()
    monkeypatch.setattr(O, "stored_h", lambda h, mode: O.dequantize_groups(
        *O.quantize_groups(np.asarray(h, np.float32), 256), 256) if mode == "fp8" else real_h(h, mode))
    assert not check_rounding_pins()
    monkeypatch.setattr(O, "stored_h", lambda h, mode: h if mode == "fp8" else real_h(h, mode))
    assert not check_rounding_pins()
    monkeypatch.setattr(O, "stored_h", real_h)
    monkeypatch.setattr(O, "stored_y", lambda y, mode: y)
    assert not check_rounding_pins()
    monkeypatch.setattr(O, "stored_y", lambda y, mode: y if mode == "fp8" else real_y(y, mode))
    assert not check_rounding_pins()
    monkeypatch.undo()
    assert check_rounding_pins()

    # dropping the renormalisation (raw softmax probabilities) breaks sum(w) = 1
    l = np.random.default_rng(1).standard_normal((4, 8)).astype(np.float32)
    p = torch.softmax(torch.from_numpy(l).double(), 1).numpy()
    ids, w = O.route(l, 2)
    raw = np.take_along_axis(p, ids.astype(np.int64), 1)
    assert not np.allclose(raw.sum(1), 1.0) and np.allclose(w.sum(1), 1.0)
