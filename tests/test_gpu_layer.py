"""moe_layer_forward end to end on the five workloads, through the C ABI, against
the C++ float64 CPU oracle.  Small cases compare every output.  Full-size workloads
compare every routing/layout integer, and the outputs of a sample of tokens built
from the layout so that it holds a token of every 128-row tile of every expert
group (the tensor-core kernels' tiles start at each group's first row), each
group's first and last rows, and a token of every 128-token tile of the shared
expert; the decode workload compares all of its tokens."""
import functools

import numpy as np
import pytest
import torch

import combine_softmax_top_expert_b300 as moe
import moe_inputs as mi
from combine_softmax_top_expert_b300.layer import Layer, PackedWeights, dtype_code
from oracle import cpp_oracle

from _util import (BF16_TOL, F32_TOL, FP8_CONSISTENCY, FP8_RMS, close, dev_f32, dev_x, fill_weights,
                   host_bf16_bits)

pytestmark = pytest.mark.gpu
O = cpp_oracle.default()


def device_generated_weights(cfg):
    """weight(which, e): the generator's logical matrix, drawn on the device and
    copied to the host (the library never touches these).  The oracle asks for each
    expert's matrices once, so only the last few are kept."""
    @functools.lru_cache(maxsize=8)
    def weight(which, e):
        t = mi.make_weight_device(cfg, which, int(e), "cuda")
        return t.cpu().numpy() if cfg.dtype == "fp32" else host_bf16_bits(t)
    return weight


def tile_sample(cfg, logits, seed=0, bias=None):
    """Tokens that cover every tile: for each physical expert group, its first and
    last rows and one random row of every 128-row tile counted from the group's
    first row; with a shared expert, one token of every 128 tokens and the last."""
    lay = O.layer_forward(cfg, logits, np.zeros((cfg.T, cfg.d), np.float32), lambda *a: None,
                          tokens=np.zeros(0, np.int64), selection_bias=bias)["layout"]
    rng = np.random.default_rng(seed)
    po, r2t = lay["phys_offsets"], lay["row_to_token"]
    toks = set()
    for p in range(len(po) - 1):
        a, b = int(po[p]), int(po[p + 1])
        if a == b:
            continue
        toks.update((int(r2t[a]), int(r2t[b - 1])))
        for s in range(a, b, 128):
            toks.add(int(r2t[rng.integers(s, min(s + 128, b))]))
    if cfg.shared:
        toks.update(int(rng.integers(s, min(s + 128, cfg.T))) for s in range(0, cfg.T, 128))
        toks.add(cfg.T - 1)
    return np.array(sorted(toks), dtype=np.int64)


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
        # the whole sample, and every sampled token on its own (a wrong tile shows up
        # in its tokens' rows)
        ratio = np.sqrt(np.mean((got - ref["out"]) ** 2)) / np.sqrt(np.mean(ref["out"] ** 2))
        per_row = np.sqrt(np.mean((got - ref["out"]) ** 2, axis=1)) / np.sqrt(np.mean(ref["out"] ** 2, axis=1))
        print(f"{cfg.name}: {len(toks)} tokens, rms error / rms(out) = {ratio:.3e} (worst token {per_row.max():.3e});"
              f" bound {FP8_RMS}")
        assert ratio <= FP8_RMS and per_row.max() <= FP8_RMS, (ratio, per_row.max())
        assert ratio <= FP8_CONSISTENCY, ratio
    elif cfg.dtype == "fp32":
        nbad, mx = close(got, ref["out"], F32_TOL)
        assert nbad == 0, (nbad, mx)
    else:
        # bf16: the kernels store every expert row y in bf16 from an fp32 sum, the
        # oracle from a float64 one; where the exact y lies near the midpoint between
        # two bf16 values the two can store different neighbours, both correct.  The
        # oracle's envelope [out_lo, out_hi] sums each y at either neighbour; the GPU
        # output must lie within the tolerance of it (the oracle's out is inside it).
        atol, rtol = BF16_TOL
        bound = atol + rtol * np.abs(ref["out"])
        excess = np.maximum(np.maximum(ref["out_lo"] - got, got - ref["out_hi"]), 0.0)
        plain = np.max(np.abs(got - ref["out"]) / bound)
        print(f"{cfg.name}: {len(toks)} tokens x {cfg.d}, largest |error| / tolerance = {plain:.3f} "
              f"(outside the bf16 envelope: {np.max(excess / bound):.3f})")
        nbad = int((excess > bound).sum())
        assert nbad == 0, (nbad, float(excess.max()))
    return layer, ref


def test_layer_tiny_fp32_full():
    check(mi.config("tiny_fp32"))


@pytest.mark.parametrize("T", [1, 3, 65])
def test_layer_tiny_fp32_ragged(T):
    check(mi.config("tiny_fp32").scaled(T=T))


def test_device_generator_matches_host():
    for workload in ("decode_bf16", "prefill_fp8_skew"):
        cfg = mi.config(workload)
        for which, e in (("w_gate", 0), ("w_down", 255)):
            dev = host_bf16_bits(mi.make_weight_device(cfg, which, e, "cuda"))
            assert np.array_equal(dev, mi.make_weight_host(cfg, which, e))
    cfg = mi.config("prefill_bf16_skew")
    dev = host_bf16_bits(mi.make_weight_device(cfg, "ws_up", 0, "cuda"))
    assert np.array_equal(dev, mi.make_weight_host(cfg, "ws_up", 0))


@pytest.mark.parametrize("kw", [dict(E=1, k=1, R=1), dict(E=8, k=8, R=4), dict(E=4, k=2, R=4, T=1)])
def test_layer_bf16_degenerate_routing(kw):
    # one expert takes every token (E = k = 1); every token takes every expert (k = E);
    # a single token
    base = dict(T=300, d=256, I=256, shared=False, zipf_bias=False)
    base.update(kw)
    check(mi.config("prefill_bf16_skew").scaled(**base))


# ------------------------------------------------------------------ bf16 workloads
def test_layer_bf16_small_full():
    check(mi.config("prefill_bf16_skew").scaled(T=200, d=256, E=16, I=256, R=4))


def test_layer_bf16_small_eplb_full():
    check(mi.config("prefill_bf16_skew_eplb").scaled(T=200, d=256, E=16, I=256, R=4, n_redundant=4))


def test_layer_bf16_small_balanced_eplb_full():
    # the load-aware placement: the hottest experts take several replicas; P % R only
    check(mi.config("prefill_bf16_skew_eplb").scaled(T=300, d=256, E=16, I=256, R=4, n_redundant=8, eplb_placement=1))


@pytest.mark.parametrize("kw", [dict(), dict(n_redundant=4), dict(n_redundant=8, eplb_placement=1)])
def test_layer_bf16_small_round_robin(kw):
    # round-robin base placement: alone (the map only renumbers), with hot-list
    # replicas, and with the load-aware map (only the "before" statistics change)
    base = dict(T=300, d=256, E=16, I=256, R=4, n_redundant=0, expert_placement=1)
    base.update(kw)
    check(mi.config("prefill_bf16_skew_eplb").scaled(**base))


@pytest.mark.parametrize("kw", [dict(), dict(shared=True, n_redundant=4)])
def test_layer_bf16_small_fp8_dispatch(kw):
    # tokens dispatched as e4m3 with per-128-channel scales, bf16 rows rebuilt for the experts
    check(mi.config("prefill_bf16_skew").scaled(T=300, d=256, E=16, I=256, R=4, shared=False, fp8_dispatch=1).scaled(**kw))


@pytest.mark.parametrize("kw", [dict(T=1), dict(T=37, d=128, I=128), dict(T=64, E=4, k=4, R=4, expert_placement=1),
                                dict(T=50, E=8, R=8, expert_placement=1), dict(T=50, E=8, R=1, expert_placement=1)])
def test_layer_bf16_edge_cases_new_options(kw):
    # one token; the smallest d and I; k = E; one expert per rank and one rank under
    # round-robin placement — with the FP8 dispatch on
    base = dict(T=300, d=256, E=16, I=256, R=4, shared=False, zipf_bias=False, fp8_dispatch=1)
    base.update(kw)
    check(mi.config("prefill_bf16_skew").scaled(**base))


@pytest.mark.parametrize("kw", [dict(T=64, E=32, k=8), dict(T=65, E=32, k=8), dict(T=32, E=64, k=8),
                                dict(T=32, E=96, k=8), dict(T=128, E=32, k=4, R=32, expert_placement=1),
                                dict(T=64, E=512, k=4, R=8), dict(T=32, E=1024, k=16, R=8)])
def test_layer_single_launch_route_and_layout_bounds(kw):
    # small batches (ceil(T/32) * k * ceil(E/32) <= 16, N <= 2048, P <= 512) are
    # routed and laid out by one launch, others by the separate kernels: both sides
    # of the bound
    base = dict(T=300, d=128, E=16, k=8, I=128, R=4, shared=False, zipf_bias=False)
    base.update(kw)
    check(mi.config("prefill_bf16_skew").scaled(**base))


def test_layer_prefill_bf16_skew_fp8_dispatch():
    cfg = mi.config("prefill_bf16_skew").scaled(fp8_dispatch=1)
    check(cfg, sample=tile_sample(cfg, mi.make_logits(cfg), seed=2))


def test_layer_fp8_experts_ignore_fp8_dispatch():
    cfg = mi.config("prefill_fp8_skew").scaled(T=300, d=256, E=8, I=256, R=4)
    a = run_layer(cfg)[3]
    b = run_layer(cfg.scaled(fp8_dispatch=1))[3]
    assert np.array_equal(a, b)


@pytest.mark.parametrize("workload,kw", [("tiny_fp32", dict()),
                                         ("prefill_bf16_skew", dict(T=300, d=256, E=16, I=256, R=4))])
def test_layer_selection_bias(workload, kw):
    # experts picked by logit + bias, weighted by the unbiased logits; the bias moves
    # the hottest expert's tokens elsewhere
    cfg = mi.config(workload).scaled(**kw)
    bias = np.linspace(-2.0, 1.0, cfg.E).astype(np.float32)
    layer, ref = check(cfg, bias=bias)
    plain = O.route(mi.make_logits(cfg), cfg.k)[0]
    assert not np.array_equal(ref["topk_ids"], plain)


def test_layer_decode_bf16():
    check(mi.config("decode_bf16"))                                   # all 128 tokens


def test_layer_prefill_bf16_skew():
    cfg = mi.config("prefill_bf16_skew")
    check(cfg, sample=tile_sample(cfg, mi.make_logits(cfg)))


def test_layer_prefill_bf16_skew_eplb():
    cfg = mi.config("prefill_bf16_skew_eplb")
    check(cfg, sample=tile_sample(cfg, mi.make_logits(cfg), seed=1))


def test_layer_prefill_bf16_skew_load_aware_eplb():
    cfg = mi.config("prefill_bf16_skew_eplb").scaled(eplb_placement=1)
    check(cfg, sample=tile_sample(cfg, mi.make_logits(cfg), seed=3))


# ------------------------------------------------------------------ fp8 workload
def test_layer_fp8_small_full():
    check(mi.config("prefill_fp8_skew").scaled(T=200, d=256, E=16, I=256, R=4))


def test_layer_prefill_fp8_skew():
    cfg = mi.config("prefill_fp8_skew")
    check(cfg, sample=tile_sample(cfg, mi.make_logits(cfg), seed=2))


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
    cfg = mi.config("prefill_bf16_skew").scaled(**{"shared": False, "zipf_bias": False, "dtype": "bf16", **kw})
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


def sweep_configs(n=16, seed=2024):
    """Seeded random small layers: every option of the layer, mixed, with ragged
    batches (bf16 experts with or without the shared expert, both EPLB placements,
    the round-robin base placement, FP8 dispatch; e4m3 experts)."""
    rng = np.random.default_rng(seed)
    cfgs = []
    for i in range(n):
        fp8 = i % 4 == 3
        E = int(rng.choice([8, 16, 32, 64]))
        R = int(rng.choice([r for r in (1, 2, 4, 8) if E % r == 0]))
        k = int(rng.integers(1, min(8, E) + 1))
        T = int(rng.integers(1, 400))
        if fp8:
            d, I, shared = int(rng.choice([256, 512])), int(rng.choice([128, 256])), False
        else:
            d, I = int(rng.choice([128, 256, 384])), int(rng.choice([128, 256, 384]))
            shared = bool(rng.integers(0, 2))
        n_red, placement = 0, 0
        if not fp8 and rng.random() < 0.5:
            placement = int(rng.integers(0, 2))
            n_red = R * int(rng.integers(1, (E // R if placement == 0 else 2 * E // R) + 1))
        cfgs.append(mi.config("prefill_bf16_skew").scaled(
            name=f"sweep{i}", T=T, d=d, E=E, k=k, I=I, R=R, shared=shared, n_redundant=n_red,
            eplb_placement=placement, expert_placement=int(rng.random() < 0.3),
            fp8_dispatch=int(not fp8 and rng.random() < 0.3), zipf_bias=bool(rng.integers(0, 2)),
            dtype="fp8" if fp8 else "bf16", seed=100 + i))
    return cfgs


SWEEP = sweep_configs()


@pytest.mark.parametrize("cfg", SWEEP, ids=[
    f"{c.name}-T{c.T}-d{c.d}-E{c.E}-k{c.k}-I{c.I}-R{c.R}-{c.dtype}{'-shared' if c.shared else ''}"
    f"{f'-eplb{c.n_redundant}p{c.eplb_placement}' if c.n_redundant else ''}{'-rr' if c.expert_placement else ''}"
    f"{'-fp8dispatch' if c.fp8_dispatch else ''}" for c in SWEEP])
def test_layer_random_small_configs(cfg):
    # every output of every token against the oracle
    check(cfg)
