"""The two fusions of the bf16 expert FFN with its neighbours.

moe_expert_gate_up_gather (the dispatch copy fused into the gate/up GEMM): h equals,
bit for bit, what moe_permute followed by moe_expert_gate_up writes on the same tiles
of 128 token rows; and the down GEMM run on that h matches the oracle's expert FFN
row by row.

moe_expert_down_combine (the combine fused into the down GEMM): y_perm equals, bit
for bit, what moe_expert_down writes on the same tiles, out equals what moe_combine
makes of it, and out matches the oracle's combine of the oracle's expert outputs."""
import os

import numpy as np
import pytest
import torch

import combine_softmax_top_expert_b300 as moe
import moe_inputs as mi
from combine_softmax_top_expert_b300.layer import PackedWeights
from oracle import moe_oracle as O

from _util import BF16_TOL, close, dev_bf16, fill_weights
from test_gpu_steps import gpu_layout

pytestmark = pytest.mark.gpu


def i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def oracle_y(cfg, xp, x, lay, p2l_np, N):
    wt = {}

    def W(which, e):
        if (which, e) not in wt:
            wt[(which, e)] = mi.f32_from_bf16_bits(mi.make_weight_host(cfg, which, e)).astype(np.float64)
        return wt[(which, e)]

    ref = np.zeros((N + (cfg.T if cfg.shared else 0), cfg.d))
    xp64 = mi.f32_from_bf16_bits(xp).astype(np.float64)
    for p in range(lay["P"]):
        a, b = lay["phys_offsets"][p], lay["phys_offsets"][p + 1]
        if b > a:
            e = p2l_np[p]
            ref[a:b] = O.swiglu_expert(xp64[a:b], W("w_gate", e), W("w_up", e), W("w_down", e), "bf16")
    if cfg.shared:
        ref[N:] = O.swiglu_expert(mi.f32_from_bf16_bits(x).astype(np.float64), W("ws_gate", 0), W("ws_up", 0),
                                  W("ws_down", 0), "bf16")
    return ref


def run_gather(cfg, logits=None, eplb=False):
    logits = mi.make_logits(cfg) if logits is None else logits
    ids, _ = O.route(logits, cfg.k)
    emap = O.eplb_map(np.bincount(ids.ravel(), minlength=cfg.E), cfg.R, cfg.n_redundant) if eplb else None
    lay = O.dispatch_layout(ids, cfg.E, cfg.R, emap)
    x = mi.make_x(cfg)
    pw = PackedWeights(cfg.E, cfg.d, cfg.I, moe.MOE_BF16, cfg.shared)
    fill_weights(cfg, pw)
    N, T_sh = cfg.N, (cfg.T if cfg.shared else 0)
    rows = N + T_sh
    xd = dev_bf16(x)
    offs = i32(lay["phys_offsets"])
    p2l = i32(emap["phys_to_logical"]) if eplb else None
    r2t = i32(lay["row_to_token"])
    s2r = i32(lay["slot_to_row"])
    sx = xd if cfg.shared else None
    err = torch.zeros(2, dtype=torch.int32, device="cuda")

    # unfused: permute, then the plain gate/up on the same one-SM tiles
    xp = torch.empty((max(N, 1), cfg.d), dtype=torch.bfloat16, device="cuda")
    moe.moe_permute(xd, moe.MOE_BF16, cfg.T, cfg.d, cfg.k, s2r, xp, moe.MOE_BF16)
    h_ref = torch.full((rows, cfg.I), float("nan"), dtype=torch.bfloat16, device="cuda")
    os.environ["MOE_B300_FFN_TILES"] = "wide"
    try:
        moe.moe_expert_gate_up(xp if N else None, None, offs, lay["P"], p2l, N, pw.struct(), sx, T_sh, h_ref,
                               None, err[0:1])
    finally:
        del os.environ["MOE_B300_FFN_TILES"]
    # fused
    h = torch.full((rows, cfg.I), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_gate_up_gather(xd, cfg.T, r2t, offs, lay["P"], p2l, N, pw.struct(), sx, T_sh, h, err[1:2])
    torch.cuda.synchronize()
    assert err.tolist() == [0, 0]
    assert torch.equal(h.view(torch.int16), h_ref.view(torch.int16))

    # the rest of the FFN on the gathered h, against the oracle
    y = torch.full((rows, cfg.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_down(h, None, offs, lay["P"], p2l, N, pw.struct(), T_sh, y, err[1:2])
    torch.cuda.synchronize()
    assert int(err[1].item()) == 0
    p2l_np = emap["phys_to_logical"] if eplb else np.arange(cfg.E)
    ref = oracle_y(cfg, O.permute(x, lay["row_to_token"]), x, lay, p2l_np, N)
    nbad, mx = close(y.float().cpu().numpy(), ref, BF16_TOL)
    assert nbad == 0, (nbad, mx)
    return lay


SMALL = mi.config("prefill_bf16_skew").scaled(T=100, d=256, E=8, I=256, R=4, shared=False, zipf_bias=False)


def test_gather_small():
    run_gather(SMALL)


def test_gather_shared_and_ragged():
    run_gather(SMALL.scaled(T=75, d=384, shared=True))


def test_gather_skewed_groups():
    # a group of several tiles with a ragged tail, empty and single-row experts
    cfg = SMALL.scaled(T=300, E=16, k=4, R=4)
    rng = np.random.default_rng(0)
    l = rng.standard_normal((cfg.T, cfg.E)).astype(np.float32)
    l[:, 3] += 6.0
    l[:, 5] -= 20.0
    run_gather(cfg, logits=l)


def test_gather_eplb_aliases_weights():
    run_gather(SMALL.scaled(T=64, E=8, k=2, R=4, n_redundant=4, zipf_bias=True), eplb=True)


def test_gather_single_token():
    run_gather(SMALL.scaled(T=1))
    run_gather(SMALL.scaled(T=1, shared=True))


def test_gather_deep_k_wraps_the_stage_ring():
    # d = 1024: 16 K blocks per tile, so the operand stages wrap within and across tiles
    cfg = mi.config("prefill_bf16_skew").scaled(T=1500, d=1024, E=32, k=8, I=512, R=4, shared=True)
    lay = run_gather(cfg)
    assert np.diff(lay["phys_offsets"]).max() > 128


def test_gather_flags_a_token_outside_x():
    # one row names token T: the kernel skips that row's copy and reports it
    cfg = SMALL.scaled(T=50)
    ids, _ = O.route(mi.make_logits(cfg), cfg.k)
    lay = O.dispatch_layout(ids, cfg.E, cfg.R, None)
    r2t = lay["row_to_token"].copy()
    r2t[7] = cfg.T
    pw = PackedWeights(cfg.E, cfg.d, cfg.I, moe.MOE_BF16, False)
    fill_weights(cfg, pw)
    h = torch.empty((cfg.N, cfg.I), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_expert_gate_up_gather(dev_bf16(mi.make_x(cfg)), cfg.T, i32(r2t), i32(lay["phys_offsets"]), lay["P"],
                                  None, cfg.N, pw.struct(), None, 0, h, err)
    torch.cuda.synchronize()
    assert int(err.item()) & moe.MOE_DEV_LAYOUT


# ------------------------------------------------------------------ fused combine
def run_combine(cfg, logits=None, eplb=False, drop_ids=0):
    logits = mi.make_logits(cfg) if logits is None else logits
    ids, tw = O.route(logits, cfg.k)
    dropped = np.zeros(ids.shape, dtype=bool)
    emap = O.eplb_map(np.bincount(ids.ravel(), minlength=cfg.E), cfg.R, cfg.n_redundant) if eplb else None
    if drop_ids:
        # ids out of range: the device layout gives those slots no row (token 0 keeps
        # none of its slots); the oracle routes them to expert 0 with weight 0
        bad = ids.copy()
        bad[:drop_ids, 0] = cfg.E + 3
        bad[0, :] = cfg.E + 5
        dropped = bad >= cfg.E
        g = gpu_layout(bad, cfg.E, cfg.R)
        assert g["err"] == moe.MOE_DEV_ID_RANGE
        lay = {"P": cfg.E, "phys_offsets": g["po"], "row_to_token": g["r2t"], "slot_to_row": g["s2r"]}
        lay_or = O.dispatch_layout(np.where(dropped, 0, ids), cfg.E, cfg.R)
    else:
        lay = lay_or = O.dispatch_layout(ids, cfg.E, cfg.R, emap)
    N = int(lay["phys_offsets"][-1])
    x = mi.make_x(cfg)
    pw = PackedWeights(cfg.E, cfg.d, cfg.I, moe.MOE_BF16, cfg.shared)
    fill_weights(cfg, pw)
    T_sh = cfg.T if cfg.shared else 0
    rows = N + T_sh
    xd = dev_bf16(x)
    offs = i32(lay["phys_offsets"])
    p2l = i32(emap["phys_to_logical"]) if eplb else None
    r2t, s2r = i32(lay["row_to_token"]), i32(lay["slot_to_row"])
    tw32 = np.ascontiguousarray(tw, dtype=np.float32)
    twd = torch.from_numpy(tw32).cuda()
    err = torch.zeros(3, dtype=torch.int32, device="cuda")
    xp = torch.empty((max(N, 1), cfg.d), dtype=torch.bfloat16, device="cuda")
    moe.moe_permute(xd, moe.MOE_BF16, cfg.T, cfg.d, cfg.k, s2r, xp, moe.MOE_BF16)
    h = torch.empty((max(rows, 1), cfg.I), dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_gate_up(xp if N else None, None, offs, lay["P"], p2l, N, pw.struct(), xd if T_sh else None,
                           T_sh, h, None, err[0:1])
    # unfused: the down GEMM on the same tiles, then the combine
    y_ref = torch.full((max(rows, 1), cfg.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    os.environ["MOE_B300_FFN_TILES"] = "wide"
    try:
        moe.moe_expert_down(h, None, offs, lay["P"], p2l, N, pw.struct(), T_sh, y_ref, err[1:2])
    finally:
        del os.environ["MOE_B300_FFN_TILES"]
    out_ref = torch.full((cfg.T, cfg.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(y_ref, moe.MOE_BF16, s2r, twd, cfg.T, cfg.k, cfg.d, y_ref[N:] if T_sh else None, out_ref,
                    moe.MOE_BF16)
    # fused
    y = torch.full_like(y_ref, float("nan"))
    out = torch.full_like(out_ref, float("nan"))
    counts = torch.full((cfg.T * (cfg.d // 128),), 12345, dtype=torch.int32, device="cuda")
    moe.moe_expert_down_combine(h, offs, lay["P"], p2l, N, pw.struct(), T_sh, r2t, s2r, twd, cfg.T, cfg.k, y,
                                counts, out, err[2:3])
    torch.cuda.synchronize()
    assert err.tolist() == [0, 0, 0]
    assert torch.equal(y[:rows].view(torch.int16), y_ref[:rows].view(torch.int16))
    assert torch.equal(out.view(torch.int16), out_ref.view(torch.int16))

    # against the oracle: its expert outputs on its own layout, combined in float64
    p2l_np = emap["phys_to_logical"] if eplb else np.arange(cfg.E)
    N_or = int(lay_or["phys_offsets"][-1])
    y_or = oracle_y(cfg, O.permute(x, lay_or["row_to_token"]), x, lay_or, p2l_np, N_or)
    w_np = np.where(dropped, 0.0, tw32.astype(np.float64))
    ref = O.combine(y_or[:N_or], lay_or["slot_to_row"], w_np, y_or[N_or:] if T_sh else None)
    nbad, mx = close(out.float().cpu().numpy(), ref, BF16_TOL)
    assert nbad == 0, (nbad, mx)
    return lay


def test_combine_small():
    run_combine(SMALL)


def test_combine_shared_ragged_and_narrow_blocks():
    # d = 384: 128-feature blocks (d is not a multiple of 256)
    run_combine(SMALL.scaled(T=75, d=384, shared=True))


def test_combine_skewed_groups():
    cfg = SMALL.scaled(T=300, E=16, k=4, R=4, shared=True)
    rng = np.random.default_rng(0)
    l = rng.standard_normal((cfg.T, cfg.E)).astype(np.float32)
    l[:, 3] += 6.0
    l[:, 5] -= 20.0
    run_combine(cfg, logits=l)


def test_combine_eplb_aliases_weights():
    run_combine(SMALL.scaled(T=64, E=8, k=2, R=4, n_redundant=4, zipf_bias=True), eplb=True)


def test_combine_slots_without_rows():
    # slots whose id is out of range have no row; token 0 has none at all (out = 0)
    run_combine(SMALL.scaled(T=40, k=2), drop_ids=5)
    run_combine(SMALL.scaled(T=40, k=2, shared=True), drop_ids=5)


def test_combine_single_token_and_k_one():
    run_combine(SMALL.scaled(T=1, shared=True))
    run_combine(SMALL.scaled(T=90, k=1))


def test_combine_many_tiles():
    cfg = mi.config("prefill_bf16_skew").scaled(T=1500, d=1024, E=32, k=8, I=512, R=4, shared=True)
    run_combine(cfg)
