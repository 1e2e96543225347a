"""moe_layer_forward end to end on the five workloads, through the C ABI, against
the CPU oracle.  Small cases compare every output; full-size workloads compare
every routing/layout integer and the outputs of a sample of tokens (the oracle
recomputes those tokens' expert rows one by one)."""
import functools

import numpy as np
import pytest
import torch

import combine_softmax_top_expert_b300 as moe
import moe_inputs as mi
from combine_softmax_top_expert_b300.layer import Layer, PackedWeights, dtype_code
from oracle import moe_oracle as O

from _util import BF16_TOL, F32_TOL, FP8_RMS, close, dev_f32, dev_x, fill_weights, host_bf16_bits

pytestmark = pytest.mark.gpu


def device_generated_weights(cfg):
    """weight(which, e): the generator's logical matrix, drawn on the device and
    copied to the host (the library never touches these)."""
    @functools.lru_cache(maxsize=None)
    def weight(which, e):
        t = mi.make_weight_device(cfg, which, int(e), "cuda")
        return t.cpu().numpy() if cfg.dtype == "fp32" else host_bf16_bits(t)
    return weight


def run_layer(cfg, bias=None):
    act = moe.MOE_F32 if cfg.dtype == "fp32" else moe.MOE_BF16
    ex = dtype_code(cfg.dtype)
    pw = PackedWeights(cfg.E, cfg.d, cfg.I, ex, cfg.shared,
                       selection_bias=None if bias is None else dev_f32(bias))
    fill_weights(cfg, pw)
    layer = Layer(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.R, act, ex, cfg.shared, cfg.n_redundant, pw,
                  eplb_placement=cfg.eplb_placement, expert_placement=cfg.expert_placement,
                  fp8_dispatch=cfg.fp8_dispatch)
    logits = mi.make_logits(cfg)
    x = mi.make_x(cfg)
    out = layer.forward(dev_f32(logits), dev_x(cfg, x))
    torch.cuda.synchronize()
    assert int(layer.err.item()) == 0
    return layer, logits, x, out.float().cpu().numpy()


def check(cfg, sample=None, bias=None):
    layer, logits, x, out = run_layer(cfg, bias)
    b = {n: t.cpu().numpy() for n, t in layer.bufs.items()}
    ref = O.layer_forward(cfg, logits, x, device_generated_weights(cfg), tokens=sample, selection_bias=bias)
    lay = ref["layout"]
    assert np.array_equal(b["topk_ids"], ref["topk_ids"])
    assert close(b["topk_w"], ref["topk_w"], F32_TOL)[0] == 0
    assert np.array_equal(b["phys_counts"], lay["phys_counts"])
    assert np.array_equal(b["phys_offsets"], lay["phys_offsets"])
    assert np.array_equal(b["rank_counts"], lay["rank_counts"])
    assert np.array_equal(b["row_to_token"], lay["row_to_token"])
    assert np.array_equal(b["slot_to_row"], lay["slot_to_row"])
    if ref["eplb"] is not None:
        em = ref["eplb"]
        assert np.array_equal(b["phys_to_logical"], em["phys_to_logical"])
        assert np.array_equal(b["replica_count"], em["replica_count"])
        assert np.array_equal(b["logical_to_phys"], em["logical_to_phys"])
    st = layer.stats()
    for s, r in zip(st, (lay["stats_before"], lay["stats_after"])):
        assert s["max_rank"] == r["max_rank"]
        assert s["max_over_mean"] == pytest.approx(r["max_over_mean"], rel=1e-6)
    toks = ref["tokens"]
    got = out[toks]
    if cfg.dtype == "fp8":
        rms = np.sqrt(np.mean((got - ref["out"]) ** 2))
        assert rms <= FP8_RMS * np.sqrt(np.mean(ref["out"] ** 2)), rms
    else:
        nbad, mx = close(got, ref["out"], F32_TOL if cfg.dtype == "fp32" else BF16_TOL)
        assert nbad == 0, (nbad, mx)
    return layer, ref


def test_layer_tiny_fp32_full():
    check(mi.config(0))


@pytest.mark.parametrize("T", [1, 3, 65])
def test_layer_tiny_fp32_ragged(T):
    check(mi.config(0).scaled(T=T))


def test_device_generator_matches_host():
    for ci in (1, 4):
        cfg = mi.config(ci)
        for which, e in (("w_gate", 0), ("w_down", 255)):
            dev = host_bf16_bits(mi.make_weight_device(cfg, which, e, "cuda"))
            assert np.array_equal(dev, mi.make_weight_host(cfg, which, e))
    cfg = mi.config(2)
    dev = host_bf16_bits(mi.make_weight_device(cfg, "ws_up", 0, "cuda"))
    assert np.array_equal(dev, mi.make_weight_host(cfg, "ws_up", 0))


@pytest.mark.parametrize("kw", [dict(E=1, k=1, R=1), dict(E=8, k=8, R=4), dict(E=4, k=2, R=4, T=1)])
def test_layer_bf16_degenerate_routing(kw):
    # one expert takes every token (E = k = 1); every token takes every expert (k = E);
    # a single token
    base = dict(T=300, d=256, I=256, shared=False, zipf_bias=False)
    base.update(kw)
    check(mi.config(2).scaled(**base))


# ------------------------------------------------------------------ bf16 workloads
def sample_tokens(T, n=6, seed=0):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, T - 1, T // 2], rng.integers(0, T, n)]))


def test_layer_bf16_small_full():
    check(mi.config(2).scaled(T=200, d=256, E=16, I=256, R=4))


def test_layer_bf16_small_eplb_full():
    check(mi.config(3).scaled(T=200, d=256, E=16, I=256, R=4, n_redundant=4))


def test_layer_bf16_small_balanced_eplb_full():
    # the load-aware placement: the hottest experts take several replicas; P % R only
    check(mi.config(3).scaled(T=300, d=256, E=16, I=256, R=4, n_redundant=8, eplb_placement=1))


@pytest.mark.parametrize("kw", [dict(), dict(n_redundant=4), dict(n_redundant=8, eplb_placement=1)])
def test_layer_bf16_small_round_robin(kw):
    # round-robin base placement: alone (the map only renumbers), with hot-list
    # replicas, and with the load-aware map (only the "before" statistics change)
    base = dict(T=300, d=256, E=16, I=256, R=4, n_redundant=0, expert_placement=1)
    base.update(kw)
    check(mi.config(3).scaled(**base))


@pytest.mark.parametrize("kw", [dict(), dict(shared=True, n_redundant=4)])
def test_layer_bf16_small_fp8_dispatch(kw):
    # tokens dispatched as e4m3 with per-128-channel scales, bf16 rows rebuilt for the experts
    check(mi.config(2).scaled(T=300, d=256, E=16, I=256, R=4, shared=False, fp8_dispatch=1).scaled(**kw))


@pytest.mark.parametrize("kw", [dict(T=1), dict(T=37, d=128, I=128), dict(T=64, E=4, k=4, R=4, expert_placement=1),
                                dict(T=50, E=8, R=8, expert_placement=1), dict(T=50, E=8, R=1, expert_placement=1)])
def test_layer_bf16_edge_cases_new_options(kw):
    # one token; the smallest d and I; k = E; one expert per rank and one rank under
    # round-robin placement — with the FP8 dispatch on
    base = dict(T=300, d=256, E=16, I=256, R=4, shared=False, zipf_bias=False, fp8_dispatch=1)
    base.update(kw)
    check(mi.config(2).scaled(**base))


@pytest.mark.parametrize("kw", [dict(T=64, E=32, k=8), dict(T=65, E=32, k=8), dict(T=32, E=64, k=8),
                                dict(T=32, E=96, k=8), dict(T=128, E=32, k=4, R=32, expert_placement=1),
                                dict(T=64, E=512, k=4, R=8), dict(T=32, E=1024, k=16, R=8)])
def test_layer_single_launch_route_and_layout_bounds(kw):
    # small batches (ceil(T/32) * k * ceil(E/32) <= 16, N <= 2048, P <= 512) are
    # routed and laid out by one launch, others by the separate kernels: both sides
    # of the bound
    base = dict(T=300, d=128, E=16, k=8, I=128, R=4, shared=False, zipf_bias=False)
    base.update(kw)
    check(mi.config(2).scaled(**base))


def test_layer_prefill_bf16_skew_fp8_dispatch():
    check(mi.config(2).scaled(fp8_dispatch=1), sample=sample_tokens(8192, n=3, seed=2))


def test_layer_fp8_experts_ignore_fp8_dispatch():
    cfg = mi.config(4).scaled(T=300, d=256, E=8, I=256, R=4)
    a = run_layer(cfg)[3]
    b = run_layer(cfg.scaled(fp8_dispatch=1))[3]
    assert np.array_equal(a, b)


@pytest.mark.parametrize("ci,kw", [(0, dict()), (2, dict(T=300, d=256, E=16, I=256, R=4))])
def test_layer_selection_bias(ci, kw):
    # experts picked by logit + bias, weighted by the unbiased logits; the bias moves
    # the hottest expert's tokens elsewhere
    cfg = mi.config(ci).scaled(**kw)
    bias = np.linspace(-2.0, 1.0, cfg.E).astype(np.float32)
    layer, ref = check(cfg, bias=bias)
    plain = O.route(mi.make_logits(cfg), cfg.k)[0]
    assert not np.array_equal(ref["topk_ids"], plain)


def test_layer_decode_bf16():
    check(mi.config(1), sample=sample_tokens(128))


def test_layer_prefill_bf16_skew():
    check(mi.config(2), sample=sample_tokens(8192, n=3))


def test_layer_prefill_bf16_skew_eplb():
    check(mi.config(3), sample=sample_tokens(8192, n=3, seed=1))


# ------------------------------------------------------------------ fp8 workload
def test_layer_fp8_small_full():
    check(mi.config(4).scaled(T=200, d=256, E=16, I=256, R=4))


def test_layer_prefill_fp8_skew():
    check(mi.config(4), sample=sample_tokens(16384, n=3, seed=2))


@pytest.mark.parametrize("name,kw", [
    ("decode-shaped bf16", dict(T=64, d=256, E=16, k=4, I=256, R=4)),
    ("prefill-shaped bf16 with shared expert and EPLB", dict(T=600, d=512, E=8, k=2, I=256, R=4, shared=True,
                                                            n_redundant=4, zipf_bias=True)),
    ("fp8", dict(T=600, d=512, E=8, k=2, I=256, R=4, dtype="fp8", zipf_bias=True)),
    ("bf16, load-aware EPLB, round-robin, FP8 dispatch, selection bias",
     dict(T=300, d=256, E=16, k=4, I=256, R=4, n_redundant=8, eplb_placement=1, expert_placement=1,
          fp8_dispatch=1, bias=True)),
])
def test_layer_forward_replays_in_a_cuda_graph(name, kw):
    """moe_layer_forward queues work on the caller's stream only (no host syncs, no
    allocation), so a CUDA graph captures it; replays on new inputs copied into the
    captured buffers give exactly what eager calls give."""
    kw = dict(kw)
    bias = kw.pop("bias", False)
    cfg = mi.config(2).scaled(**{"shared": False, "zipf_bias": False, "dtype": "bf16", **kw})
    act = moe.MOE_BF16
    ex = dtype_code(cfg.dtype)
    pw = PackedWeights(cfg.E, cfg.d, cfg.I, ex, cfg.shared,
                       selection_bias=dev_f32(np.linspace(-1, 1, cfg.E)) if bias else None)
    fill_weights(cfg, pw)
    layer = Layer(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.R, act, ex, cfg.shared, cfg.n_redundant, pw,
                  eplb_placement=cfg.eplb_placement, expert_placement=cfg.expert_placement,
                  fp8_dispatch=cfg.fp8_dispatch)
    logits_in = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
    x_in = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    batches = []
    for seed in (1, 2, 3):
        c = cfg.scaled(seed=seed)
        batches.append((dev_f32(mi.make_logits(c)), dev_x(c, mi.make_x(c))))
    eager = []
    for lg, xx in batches:
        eager.append(layer.forward(lg, xx).clone())
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):              # warm the launch paths outside the capture
        logits_in.copy_(batches[0][0])
        x_in.copy_(batches[0][1])
        layer.forward(logits_in, x_in)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = layer.forward(logits_in, x_in)
    for (lg, xx), ref in zip(batches, eager):
        logits_in.copy_(lg)
        x_in.copy_(xx)
        g.replay()
        torch.cuda.synchronize()
        assert int(layer.err.item()) == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), name
