"""GPU parity of each step of the layer against the CPU oracle, through the C ABI.
Integer results (ids, counts, offsets, rows, replica map, e4m3 codes) must match
bit for bit; floating-point results within the stated tolerances."""
import numpy as np
import pytest
import torch

import combine_softmax_top_expert_b300 as moe
import moe_inputs as mi
from combine_softmax_top_expert_b300.layer import PackedWeights
from oracle import moe_oracle as O

from _util import F32_TOL, BF16_TOL, close, dev_bf16, dev_f32, host_bf16_bits

pytestmark = pytest.mark.gpu
I32 = dict(dtype=torch.int32, device="cuda")


# ------------------------------------------------------------------ route
def gpu_route(logits, k, err=None):
    T, E = logits.shape
    L = dev_f32(logits)
    ids = torch.full((T, k), -7, **I32)
    w = torch.full((T, k), -7.0, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, **I32) if err is None else err
    moe.moe_route(L, T, E, k, ids, w, err)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy(), int(err.item())


@pytest.mark.parametrize("T,E,k", [(129, 256, 8), (64, 8, 2), (1000, 64, 6), (33, 1024, 32)])
def test_route_selection_bias(T, E, k):
    rng = np.random.default_rng(T + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    bias = (0.5 * rng.standard_normal(E)).astype(np.float32)
    bias[rng.integers(0, E)] = 3.0                   # an expert the bias pushes up
    ids = torch.full((T, k), -7, **I32)
    w = torch.full((T, k), -7.0, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, **I32)
    moe.moe_route_biased(dev_f32(logits), dev_f32(bias), T, E, k, ids, w, err)
    torch.cuda.synchronize()
    rid, rw = O.route_selection_bias(logits, bias, k)
    assert int(err.item()) == 0
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert close(w.cpu().numpy(), rw, F32_TOL)[0] == 0
    # no bias: the plain router
    moe.moe_route_biased(dev_f32(logits), None, T, E, k, ids, w, err)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), O.route(logits, k)[0])


def check_route(logits, k):
    ids, w, err = gpu_route(logits, k)
    rid, rw = O.route(logits, k)
    assert err == 0
    assert np.array_equal(ids, rid)
    nbad, mx = close(w, rw, F32_TOL)
    assert nbad == 0, mx


@pytest.mark.parametrize("workload", mi.NAMES)
def test_route_workloads(workload):
    cfg = mi.config(workload)
    check_route(mi.make_logits(cfg), cfg.k)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (3, 8, 2), (257, 33, 5), (100, 64, 32), (64, 1000, 8),
                                   (513, 256, 8), (70, 1024, 32)])
def test_route_shapes_and_ties(T, E, k):
    rng = np.random.default_rng(T * 7 + E)
    l = rng.standard_normal((T, E)).astype(np.float32)
    check_route(l, k)
    # integer logits: heavy ties resolved to the lower index; signed zeros tie
    li = rng.integers(-3, 4, size=(T, E)).astype(np.float32)
    li[li == 0] = np.where(rng.random((li == 0).sum()) < 0.5, -0.0, 0.0)
    check_route(li, k)


def test_route_flags_non_finite():
    l = np.zeros((8, 16), dtype=np.float32)
    l[3, 5] = np.nan
    l[6, 1] = np.inf
    _, _, err = gpu_route(l, 2)
    assert err & moe.MOE_DEV_NONFINITE_LOGIT


# ------------------------------------------------------------------ layout / EPLB
def gpu_layout(ids_np, E, R, eplb=None, placement="linear"):
    T, k = ids_np.shape
    P = E if eplb is None else eplb["P"]
    N = T * k
    ids = torch.from_numpy(ids_np.astype(np.int32)).cuda()
    out = {n: torch.full((m,), -9, **I32) for n, m in
           (("lc", E), ("pc", P), ("po", P + 1), ("rc", R), ("ro", R + 1), ("r2t", max(N, 1)),
            ("s2r", max(N, 1)))}
    stats = torch.zeros(16, **I32)
    wsb = moe.moe_dispatch_workspace_size(T, k, P)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, **I32)
    ep = None
    keep = []
    if eplb is not None:
        p2l = torch.from_numpy(eplb["phys_to_logical"]).cuda()
        rc = torch.from_numpy(eplb["replica_count"]).cuda()
        l2p = torch.from_numpy(eplb["logical_to_phys"]).cuda()
        keep = [p2l, rc, l2p]
        ep = moe.Eplb(P, p2l.data_ptr(), rc.data_ptr(), l2p.data_ptr(), eplb["logical_to_phys"].shape[1],
                      1 if placement == "round_robin" else 0)
    moe.moe_dispatch_layout(ids, T, k, E, R, ep, out["lc"], out["pc"], out["po"], out["rc"], out["ro"], out["r2t"],
                            out["s2r"], stats, ws, wsb, err)
    torch.cuda.synchronize()
    del keep
    res = {n: t.cpu().numpy() for n, t in out.items()}
    res["err"] = int(err.item())
    raw = stats.cpu().numpy().tobytes()
    res["stats"] = [moe.LoadStats.from_buffer_copy(raw[32 * i:32 * i + 32]) for i in range(2)]
    return res


def check_layout(ids, E, R, eplb=None, placement="linear"):
    T, k = ids.shape
    N = T * k
    g = gpu_layout(ids, E, R, eplb, placement)
    r = O.dispatch_layout(ids, E, R, eplb, placement)
    assert g["err"] == 0
    assert np.array_equal(g["lc"], r["logical_counts"])
    assert np.array_equal(g["pc"], r["phys_counts"])
    assert np.array_equal(g["po"], r["phys_offsets"])
    assert np.array_equal(g["rc"], r["rank_counts"])
    assert np.array_equal(g["ro"], r["rank_offsets"])
    assert np.array_equal(g["r2t"][:N], r["row_to_token"])
    assert np.array_equal(g["s2r"][:N], r["slot_to_row"].ravel())
    for gs, rs in zip(g["stats"], (r["stats_before"], r["stats_after"])):
        assert gs.max_rank == rs["max_rank"]
        assert gs.max_expert == rs["max_expert"]
        assert gs.n_active_experts == rs["n_active_experts"]
        assert gs.mean_rank == pytest.approx(rs["mean_rank"], rel=1e-6)
        assert gs.max_over_mean == pytest.approx(rs["max_over_mean"], rel=1e-6)
        assert gs.balancedness == pytest.approx(rs["balancedness"], rel=1e-6)
    return g, r


@pytest.mark.parametrize("workload", mi.NAMES)
def test_layout_workloads(workload):
    cfg = mi.config(workload)
    ids, _ = O.route(mi.make_logits(cfg), cfg.k)
    emap = None
    if cfg.n_redundant:
        emap = O.eplb_map(np.bincount(ids.ravel(), minlength=cfg.E), cfg.R, cfg.n_redundant)
    check_layout(ids, cfg.E, cfg.R, emap)


@pytest.mark.parametrize("T,E,k,R", [(1, 8, 2, 4), (3, 8, 2, 4), (257, 16, 4, 8), (2049, 256, 8, 64),
                                     (5000, 64, 3, 2), (300, 1024, 32, 1)])
def test_layout_shapes(T, E, k, R):
    rng = np.random.default_rng(T + E + k)
    ids, _ = O.route(rng.standard_normal((T, E)).astype(np.float32), k)
    check_layout(ids, E, R)
    # all tokens on one expert family: the most skewed histogram
    ids2, _ = O.route(np.tile(np.arange(E, dtype=np.float32)[::-1], (T, 1)), k)
    check_layout(ids2, E, R)


@pytest.mark.parametrize("T,E,R,n_red", [(64, 8, 4, 4), (777, 64, 8, 16), (4096, 256, 32, 32)])
def test_layout_with_eplb(T, E, R, n_red):
    rng = np.random.default_rng(T)
    l = rng.standard_normal((T, E)).astype(np.float32) + np.linspace(3, 0, E, dtype=np.float32)
    ids, _ = O.route(l, 4)
    emap = O.eplb_map(np.bincount(ids.ravel(), minlength=E), R, n_red)
    check_layout(ids, E, R, emap)


def test_layout_flags_out_of_range_ids():
    ids = np.array([[0, 1], [2, 9], [-1, 3]], dtype=np.int32)
    g = gpu_layout(ids, 8, 4)
    assert g["err"] & moe.MOE_DEV_ID_RANGE
    assert g["s2r"][3] == -1 and g["s2r"][4] == -1
    assert g["pc"].sum() == 4 and g["po"][-1] == 4


@pytest.mark.parametrize("E,R,n_red", [(8, 4, 4), (256, 32, 32), (256, 64, 64), (1024, 8, 8)])
def test_eplb_map(E, R, n_red):
    rng = np.random.default_rng(E + R)
    counts = rng.integers(0, 20, size=E).astype(np.int32)      # many ties
    ref = O.eplb_map(counts, R, n_red)
    P = E + n_red
    c = torch.from_numpy(counts).cuda()
    p2l, prank = torch.full((P,), -9, **I32), torch.full((P,), -9, **I32)
    rc, l2p = torch.full((E,), -9, **I32), torch.full((E, 2), -9, **I32)
    moe.moe_eplb_map(c, E, R, n_red, p2l, prank, rc, l2p)
    torch.cuda.synchronize()
    assert np.array_equal(p2l.cpu().numpy(), ref["phys_to_logical"])
    assert np.array_equal(prank.cpu().numpy(), ref["phys_rank"])
    assert np.array_equal(rc.cpu().numpy(), ref["replica_count"])
    assert np.array_equal(l2p.cpu().numpy(), ref["logical_to_phys"])


@pytest.mark.parametrize("E,R,n_red", [(8, 4, 0), (8, 4, 4), (256, 32, 0), (256, 32, 32), (1024, 8, 8), (12, 3, 6)])
def test_placement_map_round_robin(E, R, n_red):
    rng = np.random.default_rng(E * 7 + R)
    counts = rng.integers(0, 20, size=E).astype(np.int32)
    ref = O.eplb_map(counts, R, n_red, "round_robin")
    P = E + n_red
    c = torch.from_numpy(counts).cuda() if n_red else None       # the bare placement reads no counts
    p2l, prank = torch.full((P,), -9, **I32), torch.full((P,), -9, **I32)
    rc, l2p = torch.full((E,), -9, **I32), torch.full((E, 2), -9, **I32)
    moe.moe_placement_map(c, E, R, n_red, 1, p2l, prank, rc, l2p)
    torch.cuda.synchronize()
    assert np.array_equal(p2l.cpu().numpy(), ref["phys_to_logical"])
    assert np.array_equal(prank.cpu().numpy(), ref["phys_rank"])
    assert np.array_equal(rc.cpu().numpy(), ref["replica_count"])
    assert np.array_equal(l2p.cpu().numpy(), ref["logical_to_phys"])
    # placement 0 is moe_eplb_map
    if n_red:
        lin = O.eplb_map(counts, R, n_red)
        moe.moe_placement_map(c, E, R, n_red, 0, p2l, prank, rc, l2p)
        torch.cuda.synchronize()
        assert np.array_equal(p2l.cpu().numpy(), lin["phys_to_logical"])
        assert np.array_equal(l2p.cpu().numpy(), lin["logical_to_phys"])


@pytest.mark.parametrize("T,E,R,n_red", [(64, 8, 4, 0), (777, 64, 8, 16), (4096, 256, 32, 0), (4096, 256, 32, 32)])
def test_layout_round_robin(T, E, R, n_red):
    rng = np.random.default_rng(T + 1)
    l = rng.standard_normal((T, E)).astype(np.float32) + np.linspace(3, 0, E, dtype=np.float32)
    ids, _ = O.route(l, 4)
    emap = O.eplb_map(np.bincount(ids.ravel(), minlength=E), R, n_red, "round_robin")
    check_layout(ids, E, R, emap, "round_robin")
    # the load-aware map with round-robin "before" statistics
    if n_red:
        check_layout(ids, E, R, O.eplb_balanced_map(np.bincount(ids.ravel(), minlength=E), R, n_red),
                     "round_robin")


# ------------------------------------------------------------------ FP8 dispatch, receive side
@pytest.mark.parametrize("rows,d", [(1, 128), (37, 384), (4096, 7168), (3, 640)])
def test_dequantize_e4m3_exact(rows, d):
    rng = np.random.default_rng(rows + d)
    codes = rng.integers(0, 256, size=(rows, d)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x7E                          # the quantiser makes no NaN codes
    if d >= 256:
        codes[0, :256] = np.where((np.arange(256) & 0x7F) == 0x7F, 0, np.arange(256)).astype(np.uint8)
    scales = (2.0 ** rng.uniform(-20, 20, size=(rows, d // 128))).astype(np.float32)
    out = torch.empty((rows, d), dtype=torch.bfloat16, device="cuda")
    moe.moe_dequantize_e4m3(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(), rows, d, out)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.array_equal(got, O.dequantize_groups_bf16(codes, scales))


@pytest.mark.parametrize("T,d", [(300, 256), (8192, 7168)])
def test_fp8_dispatch_round_trip(T, d):
    """permute to e4m3 then the receive side, against the oracle's quantise + dequantise."""
    rng = np.random.default_rng(T)
    k = 4
    ids, _ = O.route(rng.standard_normal((T, 16)).astype(np.float32), k)
    lay = O.dispatch_layout(ids, 16, 4)
    xb = torch.randn((T, d), generator=torch.Generator().manual_seed(T)).bfloat16()
    N = T * k
    xq = torch.empty((N, d), dtype=torch.uint8, device="cuda")
    xs = torch.empty((N, d // 128), dtype=torch.float32, device="cuda")
    xr = torch.empty((N, d), dtype=torch.bfloat16, device="cuda")
    s2r = torch.from_numpy(lay["slot_to_row"].astype(np.int32)).cuda()
    moe.moe_permute(xb.cuda(), moe.MOE_BF16, T, d, k, s2r, xq, moe.MOE_E4M3, xs)
    moe.moe_dequantize_e4m3(xq, xs, N, d, xr)
    torch.cuda.synchronize()
    q, sc = O.quantize_groups(xb.float().numpy())
    want = O.dequantize_groups_bf16(q, sc)[lay["row_to_token"]]
    assert np.array_equal(xr.float().cpu().numpy().astype(np.float64), want)


# ------------------------------------------------------------------ permute / combine
def layout_for(cfg):
    ids, w = O.route(mi.make_logits(cfg), cfg.k)
    return ids, w, O.dispatch_layout(ids, cfg.E, cfg.R)


def gpu_balanced_map(counts, R, n_red):
    E = counts.size
    P = E + n_red
    c = torch.from_numpy(counts.astype(np.int32)).cuda()
    p2l = torch.full((P,), -9, **I32)
    prank = torch.full((P,), -9, **I32)
    rc = torch.full((E,), -9, **I32)
    l2p = torch.full((E, 1 + n_red), -9, **I32)
    load = torch.full((R,), -1.0, dtype=torch.float64, device="cuda")
    moe.moe_eplb_balanced_map(c, E, R, n_red, p2l, prank, rc, l2p, load)
    torch.cuda.synchronize()
    return {"phys_to_logical": p2l.cpu().numpy(), "phys_rank": prank.cpu().numpy(),
            "replica_count": rc.cpu().numpy(), "logical_to_phys": l2p.cpu().numpy(),
            "rank_load": load.cpu().numpy(), "P": P}


@pytest.mark.parametrize("E,R,n_red,seed", [(256, 8, 0, 0), (256, 32, 32, 1), (256, 64, 64, 2), (256, 256, 256, 3),
                                            (64, 4, 12, 4), (1024, 64, 1024, 5), (8, 3, 1, 6)])
def test_eplb_balanced_map_exact(E, R, n_red, seed):
    rng = np.random.default_rng(seed)
    counts = rng.integers(0, 300, size=E)
    counts[rng.integers(0, E, size=3)] = 5000        # hot experts that need several replicas
    counts[:4] = counts[4]                           # ties, broken by expert id
    g = gpu_balanced_map(counts, R, n_red)
    r = O.eplb_balanced_map(counts, R, n_red)
    for key in ("phys_to_logical", "phys_rank", "replica_count", "logical_to_phys"):
        assert np.array_equal(g[key], r[key]), key
    assert np.array_equal(g["rank_load"], r["rank_load"])   # fp64, same operations in the same order


def test_eplb_balanced_map_worked_examples():
    """The hand-worked placements of the oracle's pins, through the GPU map."""
    g = gpu_balanced_map(np.array([10, 6, 3, 1]), 2, 2)
    assert g["phys_to_logical"].tolist() == [0, 1, 2, 0, 1, 3]
    assert g["logical_to_phys"].tolist() == [[0, 3, -1], [1, 4, -1], [2, -1, -1], [5, -1, -1]]
    assert g["rank_load"].tolist() == [11.0, 9.0]
    g = gpu_balanced_map(np.array([100, 1, 1, 1]), 2, 2)
    assert g["replica_count"].tolist() == [3, 1, 1, 1]
    assert g["phys_to_logical"].tolist() == [0, 0, 3, 0, 1, 2]
    assert g["rank_load"].tolist() == [100 / 3 + 100 / 3 + 1.0, 100 / 3 + 1.0 + 1.0]
    # one expert per card: nothing to move, the busiest card keeps the hottest expert
    counts = np.full(256, 125)
    counts[17] = 640
    counts[18] = 128 * 256 - 640 - 125 * 254
    g = gpu_balanced_map(counts, 256, 0)
    assert round(g["rank_load"].max() / g["rank_load"].mean(), 2) == 5.0


@pytest.mark.parametrize("W,E", [(3, 8), (1, 256), (5, 256)])
def test_eplb_window_then_balanced_map(W, E):
    """Per-step counts through the device ring; each step's window sum, and the
    load-aware map built on it, equal the oracle's."""
    rng = np.random.default_rng(W + E)
    ring = torch.zeros((W, E), **I32)
    wsum = torch.full((E,), -1, **I32)
    history = []
    for step in range(7):
        counts = rng.integers(0, 500, size=E).astype(np.int32)
        counts[step % E] += 3000                      # a hot expert that moves
        history.append(counts)
        moe.moe_eplb_window_update(torch.from_numpy(counts).cuda(), ring, W, E, step, wsum)
        torch.cuda.synchronize()
        ref = O.eplb_window_sum(history, W)
        assert np.array_equal(wsum.cpu().numpy(), ref)
    g = gpu_balanced_map(ref, 8, 8)
    r = O.eplb_balanced_map(ref, 8, 8)
    assert np.array_equal(g["logical_to_phys"], r["logical_to_phys"])
    assert np.array_equal(g["rank_load"], r["rank_load"])


@pytest.mark.parametrize("T,E,R,n_red", [(300, 16, 4, 4), (2048, 64, 8, 24), (8192, 256, 32, 32)])
def test_layout_with_balanced_map(T, E, R, n_red):
    rng = np.random.default_rng(T)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[:, : E // 8] += 2.0                        # a hot block of experts
    ids, _ = O.route(logits, 4)
    emap = O.eplb_balanced_map(np.bincount(ids.ravel(), minlength=E), R, n_red)
    check_layout(ids, E, R, emap)


@pytest.mark.parametrize("workload,T", [("tiny_fp32", None), ("decode_bf16", None), ("prefill_bf16_skew", 1024),
                                        ("prefill_fp8_skew", 512)])
def test_permute_copy_is_exact(workload, T):
    cfg = mi.config(workload) if T is None else mi.config(workload).scaled(T=T)
    ids, w, lay = layout_for(cfg)
    x = mi.make_x(cfg)
    dt = moe.MOE_F32 if cfg.dtype == "fp32" else moe.MOE_BF16
    xd = dev_f32(x) if cfg.dtype == "fp32" else dev_bf16(x)
    s2r = torch.from_numpy(lay["slot_to_row"].astype(np.int32)).cuda()
    xp = torch.zeros((cfg.N, cfg.d), dtype=xd.dtype, device="cuda")
    moe.moe_permute(xd, dt, cfg.T, cfg.d, cfg.k, s2r, xp, dt)
    torch.cuda.synchronize()
    ref = O.permute(x, lay["row_to_token"])
    got = xp.cpu().numpy() if cfg.dtype == "fp32" else host_bf16_bits(xp)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("T,d", [(16384, 6144), (37, 128), (5, 384)])
def test_permute_e4m3_codes_exact(T, d):
    cfg = mi.config("prefill_fp8_skew").scaled(T=T, d=d)
    ids, w, lay = layout_for(cfg)
    x = mi.make_x(cfg)
    # add scale variety and exact zeros per group
    xf = mi.f32_from_bf16_bits(x) * np.float32(7.5)
    xf[1 % T, :128] = 0.0
    x = mi.bf16_bits_from_f32(xf)
    s2r = torch.from_numpy(lay["slot_to_row"].astype(np.int32)).cuda()
    xq = torch.zeros((cfg.N, d), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((cfg.N, d // 128), dtype=torch.float32, device="cuda")
    moe.moe_permute(dev_bf16(x), moe.MOE_BF16, T, d, cfg.k, s2r, xq, moe.MOE_E4M3, sc)
    torch.cuda.synchronize()
    q, s = O.quantize_groups(mi.f32_from_bf16_bits(x))
    r2t = lay["row_to_token"]
    assert np.array_equal(xq.cpu().numpy(), q[r2t])
    assert np.array_equal(sc.cpu().numpy(), s[r2t])


@pytest.mark.parametrize("workload,T", [("tiny_fp32", None), ("decode_bf16", None), ("prefill_bf16_skew", 2048)])
def test_combine_and_identity_experts(workload, T):
    cfg = mi.config(workload) if T is None else mi.config(workload).scaled(T=T)
    ids, w, lay = layout_for(cfg)
    rng = np.random.default_rng(mi.NAMES.index(workload))
    y = rng.standard_normal((cfg.N, cfg.d)).astype(np.float32)
    sh = rng.standard_normal((cfg.T, cfg.d)).astype(np.float32)
    dt = moe.MOE_F32 if cfg.dtype == "fp32" else moe.MOE_BF16
    if dt == moe.MOE_BF16:
        yb, shb = mi.bf16_bits_from_f32(y), mi.bf16_bits_from_f32(sh)
        y, sh = mi.f32_from_bf16_bits(yb), mi.f32_from_bf16_bits(shb)
        yd, shd = dev_bf16(yb), dev_bf16(shb)
        tol = BF16_TOL
    else:
        yd, shd, tol = dev_f32(y), dev_f32(sh), F32_TOL
    s2r = torch.from_numpy(lay["slot_to_row"].astype(np.int32)).cuda()
    tw = dev_f32(w)
    out = torch.empty((cfg.T, cfg.d), dtype=yd.dtype, device="cuda")
    for shared in (None, shd):
        moe.moe_combine(yd, dt, s2r, tw, cfg.T, cfg.k, cfg.d, shared, out, dt)
        torch.cuda.synchronize()
        ref = O.combine(y.astype(np.float64), lay["slot_to_row"], w, None if shared is None else sh)
        got = out.float().cpu().numpy()
        nbad, mx = close(got, ref, tol)
        assert nbad == 0, mx
    # identity experts: y = x_perm, weights renormalised -> out = x
    x = mi.make_x(cfg)
    xd = dev_f32(x) if dt == moe.MOE_F32 else dev_bf16(x)
    xp = torch.empty((cfg.N, cfg.d), dtype=xd.dtype, device="cuda")
    moe.moe_permute(xd, dt, cfg.T, cfg.d, cfg.k, s2r, xp, dt)
    moe.moe_combine(xp, dt, s2r, tw, cfg.T, cfg.k, cfg.d, None, out, dt)
    torch.cuda.synchronize()
    xf = x if dt == moe.MOE_F32 else mi.f32_from_bf16_bits(x)
    nbad, mx = close(out.float().cpu().numpy(), xf, (1e-6, 1e-6) if dt == moe.MOE_F32 else (0.0, 2 ** -8))
    assert nbad == 0, mx


# ------------------------------------------------------------------ weight packing
def tiled(m, rows_per_tile=128):
    """The packed layout of a K-major matrix m [rows, K] (uint16 or uint8):
    rows_per_tile x 128-byte blocks, tile major then column block, the 16-byte
    chunk j of block row r moved to j ^ (r % 8)."""
    b = np.ascontiguousarray(m).view(np.uint8)
    rows, nb = b.shape
    t = b.reshape(rows // rows_per_tile, rows_per_tile, nb // 128, 8, 16)
    out = np.empty_like(t)
    for r in range(rows_per_tile):
        for j in range(8):
            out[:, r, :, j ^ (r % 8), :] = t[:, r, :, j, :]
    return out.transpose(0, 2, 1, 3, 4).reshape(-1)


def gate_up_interleaved(g_t, u_t):
    """W_gate^T and W_up^T rows in 256-row tiles: the gate rows then the up rows of
    each group of 128 features."""
    I = g_t.shape[0]
    parts = []
    for f in range(0, I, 128):
        parts += [g_t[f:f + 128], u_t[f:f + 128]]
    return np.concatenate(parts)


def packed_bytes(t):
    return t.contiguous().view(torch.uint8).cpu().numpy().reshape(-1)


@pytest.mark.parametrize("dst", ["bf16", "fp8", "fp32"])
def test_pack_weights(dst):
    d, I = 256, 384
    cfg = mi.config("decode_bf16").scaled(d=d, I=I, dtype="fp32" if dst == "fp32" else "bf16")
    code = {"bf16": moe.MOE_BF16, "fp8": moe.MOE_E4M3, "fp32": moe.MOE_F32}[dst]
    pw = PackedWeights(2, d, I, code, False)
    wg, wu, wd = (mi.make_weight_host(cfg, n, 1) for n in ("w_gate", "w_up", "w_down"))
    devw = [dev_f32(a) if dst == "fp32" else dev_bf16(a) for a in (wg, wu, wd)]
    pw.pack(1, *devw)
    torch.cuda.synchronize()
    if dst == "fp32":
        assert np.array_equal(pw.w13[1].cpu().numpy(), np.concatenate([wg.T, wu.T]))
        assert np.array_equal(pw.w2[1].cpu().numpy(), wd.T)
    elif dst == "bf16":
        assert np.array_equal(packed_bytes(pw.w13[1]), tiled(gate_up_interleaved(wg.T, wu.T), 256))
        assert np.array_equal(packed_bytes(pw.w2[1]), tiled(wd.T))
    else:
        f = [mi.f32_from_bf16_bits(a) for a in (wg, wu, wd)]
        qs = [O.quantize_blocks(a) for a in f]
        assert np.array_equal(packed_bytes(pw.w13[1]), tiled(gate_up_interleaved(qs[0][0].T, qs[1][0].T), 256))
        assert np.array_equal(packed_bytes(pw.w2[1]), tiled(qs[2][0].T))
        assert np.array_equal(pw.s13[1].cpu().numpy(), np.concatenate([qs[0][1].T, qs[1][1].T]))
        assert np.array_equal(pw.s2[1].cpu().numpy(), qs[2][1].T)
