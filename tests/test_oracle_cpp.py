"""The C++ float64 oracle against the numpy one (no GPU): on the five workloads
(scaled down) and their options, every integer output is identical and every float
agrees to 1e-12 relative; then each planted mistake, compiled into its own build of
the C++ oracle, makes one of the pins fail."""
import functools
import os
import sys
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import moe_inputs as mi
from oracle import build as orc_build
from oracle import cpp_oracle
from oracle import moe_oracle as NP

CPP = cpp_oracle.default()


def host_weights(cfg):
    @functools.lru_cache(maxsize=None)
    def weight(which, e):
        return mi.make_weight_host(cfg, which, int(e))
    return weight


def assert_same_layer(a, b):
    assert np.array_equal(a["topk_ids"], b["topk_ids"])
    np.testing.assert_allclose(b["topk_w"], a["topk_w"], rtol=1e-12, atol=0)
    for key, va in a["layout"].items():
        vb = b["layout"][key]
        if isinstance(va, dict):
            for kk in va:
                assert vb[kk] == pytest.approx(va[kk], rel=1e-12, abs=0), (key, kk)
        else:
            assert np.array_equal(np.asarray(va), np.asarray(vb)), key
    assert (a["eplb"] is None) == (b["eplb"] is None)
    if a["eplb"] is not None:
        for key, va in a["eplb"].items():
            assert np.array_equal(np.asarray(va), np.asarray(b["eplb"][key])), key
    scale = max(float(np.abs(a["out"]).max()), 1e-300)
    for key in ("out", "out_lo", "out_hi"):
        assert np.abs(a[key] - b[key]).max() <= 1e-12 * scale, key
    if "x_q" in a:
        assert np.array_equal(a["x_q"], b["x_q"]) and np.array_equal(a["x_scales"], b["x_scales"])
    if a["out_rounded"] is a["out"]:                     # fp32 workload: nothing rounded
        return
    # bf16-rounded outputs can differ only where the two float64 sums straddle a
    # rounding boundary: at most one bf16 step, and rarely
    diff = a["out_rounded"] != b["out_rounded"]
    assert diff.mean() <= 1e-3
    if diff.any():
        step = np.abs(a["out_rounded"][diff]) * 2.0 ** -7
        assert np.all(np.abs(a["out_rounded"][diff] - b["out_rounded"][diff]) <= step * (1 + 1e-9))


CASES = [
    ("tiny_fp32", "tiny_fp32", dict()),
    ("tiny_fp32, round-robin", "tiny_fp32", dict(expert_placement=1)),
    ("tiny_fp32, ragged", "tiny_fp32", dict(T=37)),
    ("decode-shaped bf16", "decode_bf16", dict(d=256, I=256, E=32, R=8)),
    ("prefill bf16 + shared", "prefill_bf16_skew", dict(T=300, d=256, E=16, I=256, R=4)),
    ("prefill bf16 + EPLB", "prefill_bf16_skew_eplb", dict(T=300, d=256, E=16, I=256, R=4, n_redundant=4)),
    ("prefill bf16 + load-aware EPLB", "prefill_bf16_skew_eplb",
     dict(T=300, d=256, E=16, I=256, R=4, n_redundant=8, eplb_placement=1)),
    ("prefill bf16 + EPLB, round-robin", "prefill_bf16_skew_eplb",
     dict(T=300, d=256, E=16, I=256, R=4, n_redundant=4, expert_placement=1)),
    ("prefill bf16, FP8 dispatch", "prefill_bf16_skew", dict(T=300, d=256, E=16, I=256, R=4, fp8_dispatch=1)),
    ("fp8 experts", "prefill_fp8_skew", dict(T=300, d=256, E=16, I=256, R=4)),
    ("degenerate E = k = 1", "prefill_bf16_skew", dict(T=50, d=128, E=1, k=1, I=128, R=1, shared=False)),
    ("k = E", "prefill_bf16_skew", dict(T=50, d=128, E=8, k=8, I=128, R=4, shared=False)),
]


@pytest.mark.parametrize("name,workload,kw", CASES, ids=[c[0] for c in CASES])
def test_cpp_layer_equals_numpy(name, workload, kw):
    cfg = mi.config(workload).scaled(**kw)
    logits, x = mi.make_logits(cfg), mi.make_x(cfg)
    w = host_weights(cfg)
    a = NP.layer_forward(cfg, logits, x, w)
    b = CPP.layer_forward(cfg, logits, x, w)
    assert_same_layer(a, b)
    assert set(b["seconds"]) == set(cpp_oracle.STEPS)


def test_cpp_layer_token_subset_and_selection_bias():
    cfg = mi.config("prefill_bf16_skew").scaled(T=300, d=256, E=16, I=256, R=4)
    logits, x = mi.make_logits(cfg), mi.make_x(cfg)
    w = host_weights(cfg)
    toks = np.array([0, 7, 150, 299])
    bias = np.linspace(-2.0, 1.0, cfg.E).astype(np.float32)
    for kw in (dict(tokens=toks), dict(selection_bias=bias), dict(tokens=toks, selection_bias=bias)):
        assert_same_layer(NP.layer_forward(cfg, logits, x, w, **kw), CPP.layer_forward(cfg, logits, x, w, **kw))
    full = CPP.layer_forward(cfg, logits, x, w)
    part = CPP.layer_forward(cfg, logits, x, w, tokens=toks)
    assert np.array_equal(full["out"][toks], part["out"])     # rows are computed one by one


def test_cpp_layer_threads_do_not_change_results():
    cfg = mi.config("prefill_fp8_skew").scaled(T=300, d=256, E=16, I=256, R=4)
    logits, x = mi.make_logits(cfg), mi.make_x(cfg)
    w = host_weights(cfg)
    one = CPP.layer_forward(cfg, logits, x, w, threads=1)
    many = CPP.layer_forward(cfg, logits, x, w, threads=7)
    assert np.array_equal(one["out"], many["out"])


def test_cpp_layer_rejects_bad_input():
    cfg = mi.config("tiny_fp32")
    logits, x = mi.make_logits(cfg), mi.make_x(cfg)
    logits[3, 1] = np.inf
    with pytest.raises(ValueError):
        CPP.layer_forward(cfg, logits, x, host_weights(cfg))
    with pytest.raises(ValueError):
        CPP.layer_forward(cfg, mi.make_logits(cfg), x, host_weights(cfg), tokens=np.array([3, 2]))


def test_cpp_balanced_map_equals_numpy_on_random_counts():
    rng = np.random.default_rng(31)
    for E, R, n_red in ((256, 32, 32), (256, 64, 64), (64, 8, 40), (30, 4, 10), (8, 3, 1), (1024, 64, 1024)):
        for trial in range(4):
            counts = rng.integers(0, 400 if trial % 2 else 4, size=E)
            counts[rng.integers(0, E, 3)] = 9000
            a, b = NP.eplb_balanced_map(counts, R, n_red), CPP.eplb_balanced_map(counts, R, n_red)
            for key in a:
                assert np.array_equal(np.asarray(a[key]), np.asarray(b[key])), (E, R, n_red, key)


# ------------------------------------------------------------------ planted mistakes
PLANTS = {
    1: ("ties to the higher expert index", "test_route_brute_force_with_ties", dict(E=6, k=3)),
    2: ("weights not renormalised over the k", "test_route_weights_two_forms_agree", {}),
    3: ("sign slip in silu", "test_ffn_single_expert_is_dense_swiglu", {}),
    4: ("h not rounded to bf16", "test_bf16_mode_rounds_h_at_a_tie", {}),
    5: ("h quantised over 256 channels", "test_fp8_mode_quantises_h_per_128_channels", {}),
    6: ("h not quantised in the fp8 mode", "test_fp8_mode_quantises_h_per_128_channels", {}),
    7: ("y not rounded to bf16", "test_bf16_mode_rounds_y", {}),
    8: ("gate and up exchanged", "test_ffn_single_expert_is_dense_swiglu", {}),
}


@pytest.fixture(scope="module")
def planted(tmp_path_factory):
    d = tmp_path_factory.mktemp("planted")
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        paths = dict(zip(PLANTS, ex.map(lambda n: orc_build.build(str(d / f"libplant{n}.so"), plant=n, force=True),
                                        PLANTS)))
    return {n: cpp_oracle.CppOracle(p) for n, p in paths.items()}


@pytest.mark.parametrize("n", sorted(PLANTS), ids=[PLANTS[n][0] for n in sorted(PLANTS)])
def test_cpp_planted_mistake_fails_a_pin(n, planted, monkeypatch):
    sys.path.insert(0, os.path.dirname(__file__))
    import test_oracle_pins as pins

    _, pin_name, kw = PLANTS[n]
    pin = getattr(pins, pin_name)
    assert planted[n].plant == n
    monkeypatch.setattr(pins, "O", CPP)           # the default build passes the pin
    pin(**kw)
    monkeypatch.setattr(pins, "O", planted[n])    # the planted build fails it
    with pytest.raises(AssertionError):
        pin(**kw)
