"""Grouped SwiGLU expert FFN (moe_expert_ffn) against the oracle, every output row,
in every tile orientation of the tensor-core kernels (swap, wide, SM pair)."""
import os

import numpy as np
import pytest
import torch

import combine_softmax_top_expert_b300 as moe
import moe_inputs as mi
from combine_softmax_top_expert_b300.layer import PackedWeights
from oracle import moe_oracle as O

from _util import BF16_TOL, close, dev_bf16, fill_weights, host_bf16_bits

pytestmark = pytest.mark.gpu


def run_ffn(cfg, mode, logits=None, eplb=False):
    """Route/lay out on the host (oracle), run moe_expert_ffn on the GPU, compare
    y_perm row by row with the oracle's expert FFN."""
    logits = mi.make_logits(cfg) if logits is None else logits
    ids, w = O.route(logits, cfg.k)
    emap = O.eplb_map(np.bincount(ids.ravel(), minlength=cfg.E), cfg.R, cfg.n_redundant) if eplb else None
    lay = O.dispatch_layout(ids, cfg.E, cfg.R, emap)
    x = mi.make_x(cfg)
    xp = O.permute(x, lay["row_to_token"])
    pw = PackedWeights(cfg.E, cfg.d, cfg.I, moe.MOE_BF16, cfg.shared)
    fill_weights(cfg, pw)
    N, T_sh = cfg.N, (cfg.T if cfg.shared else 0)
    rows = N + T_sh
    y = torch.full((rows, cfg.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    wsb = moe.moe_ffn_workspace_size(rows, cfg.I, moe.MOE_BF16)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    offs = torch.from_numpy(lay["phys_offsets"].astype(np.int32)).cuda()
    p2l = torch.from_numpy(emap["phys_to_logical"]).cuda() if eplb else None
    xd = dev_bf16(xp) if N else None
    sx = dev_bf16(x) if cfg.shared else None
    os.environ["MOE_B300_FFN_TILES"] = mode
    try:
        moe.moe_expert_ffn(xd, None, offs, lay["P"], p2l, N, pw.struct(), sx, T_sh, y, ws, wsb, err)
        torch.cuda.synchronize()
    finally:
        del os.environ["MOE_B300_FFN_TILES"]
    assert int(err.item()) == 0
    got = y.float().cpu().numpy()
    wt = {}

    def W(which, e):
        if (which, e) not in wt:
            wt[(which, e)] = mi.f32_from_bf16_bits(mi.make_weight_host(cfg, which, e)).astype(np.float64)
        return wt[(which, e)]

    p2l_np = emap["phys_to_logical"] if eplb else np.arange(cfg.E)
    ref = np.zeros((rows, cfg.d))
    xp64 = mi.f32_from_bf16_bits(xp).astype(np.float64)
    for p in range(lay["P"]):
        a, b = lay["phys_offsets"][p], lay["phys_offsets"][p + 1]
        if b > a:
            e = p2l_np[p]
            ref[a:b] = O.swiglu_expert(xp64[a:b], W("w_gate", e), W("w_up", e), W("w_down", e), "bf16")
    if cfg.shared:
        ref[N:] = O.swiglu_expert(mi.f32_from_bf16_bits(x).astype(np.float64), W("ws_gate", 0), W("ws_up", 0),
                                  W("ws_down", 0), "bf16")
    nbad, mx = close(got, ref, BF16_TOL)
    assert nbad == 0, (nbad, mx)
    return lay


SMALL = mi.config("prefill_bf16_skew").scaled(T=100, d=256, E=8, I=256, R=4, shared=False, zipf_bias=False)


@pytest.mark.parametrize("mode", ["swap", "wide", "pair"])
def test_ffn_small(mode):
    run_ffn(SMALL, mode)


@pytest.mark.parametrize("mode", ["swap", "wide", "pair"])
def test_ffn_shared_and_ragged(mode):
    # d = 384 is not a multiple of 256: the wide down GEMM takes 128-feature tiles
    # and the pair down GEMM hands over to it
    run_ffn(SMALL.scaled(T=75, d=384, shared=True), mode)


@pytest.mark.parametrize("mode", ["swap", "wide", "pair"])
def test_ffn_skewed_groups(mode):
    # one expert gets almost every token: a group of many tiles with a ragged tail,
    # plus empty experts and single-row experts
    cfg = SMALL.scaled(T=300, E=16, k=4, R=4)
    rng = np.random.default_rng(0)
    l = rng.standard_normal((cfg.T, cfg.E)).astype(np.float32)
    l[:, 3] += 6.0
    l[:, 5] -= 20.0
    run_ffn(cfg, mode, logits=l)


@pytest.mark.parametrize("mode", ["swap", "wide", "pair"])
def test_ffn_eplb_aliases_weights(mode):
    cfg = SMALL.scaled(T=64, E=8, k=2, R=4, n_redundant=4, zipf_bias=True)
    run_ffn(cfg, mode, eplb=True)


def test_ffn_single_token():
    run_ffn(SMALL.scaled(T=1), "swap")
    run_ffn(SMALL.scaled(T=1), "wide")
    run_ffn(SMALL.scaled(T=1), "pair")


def test_ffn_pair_tile_edges():
    # three feature tiles per expert and groups from empty to several 256-row pair
    # tiles, so the odd SM's half of a tile is full, partly filled or empty
    cfg = SMALL.scaled(T=700, d=512, E=8, k=2, I=384, R=4)
    rng = np.random.default_rng(1)
    l = rng.standard_normal((cfg.T, cfg.E)).astype(np.float32)
    l[:, 1] += 3.0
    l[:, 6] -= 20.0
    lay = run_ffn(cfg, "pair", logits=l)
    counts = np.diff(lay["phys_offsets"])
    assert counts.max() > 512 and (counts == 0).any()


@pytest.mark.parametrize("mode", ["swap", "wide", "pair"])
def test_ffn_smallest_dims(mode):
    # d = I = 128: one K block and one feature tile in every GEMM (d < 256, so the pair
    # orientation's down projection runs on one-SM tiles)
    run_ffn(SMALL.scaled(T=50, d=128, I=128, E=4, k=2, R=2, shared=True), mode)


@pytest.mark.parametrize("eplb", [False, True], ids=["linear", "eplb"])
@pytest.mark.parametrize("mode", ["swap", "wide", "pair"])
def test_ffn_per_rank_slices_equal_the_whole(mode, eplb):
    # the layout orders rows by (rank, expert): each logical rank's slice of x_perm,
    # with its own experts' offsets, runs on its own and gives exactly the rows the
    # whole batch gives them -- what an expert-parallel deployment would run per GPU
    cfg = SMALL.scaled(T=300, E=16, k=4, R=4, n_redundant=4 if eplb else 0, zipf_bias=True)
    ids, _ = O.route(mi.make_logits(cfg), cfg.k)
    emap = O.eplb_map(np.bincount(ids.ravel(), minlength=cfg.E), cfg.R, cfg.n_redundant) if eplb else None
    lay = O.dispatch_layout(ids, cfg.E, cfg.R, emap)
    P, N = lay["P"], cfg.N
    p2l_all = emap["phys_to_logical"] if eplb else np.arange(P, dtype=np.int32)
    po = lay["phys_offsets"].astype(np.int64)
    xp = dev_bf16(O.permute(mi.make_x(cfg), lay["row_to_token"]))
    pw = PackedWeights(cfg.E, cfg.d, cfg.I, moe.MOE_BF16, False)
    fill_weights(cfg, pw)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def ffn(x_rows, offs, n_phys, p2l, rows):
        y = torch.full((max(rows, 1), cfg.d), float("nan"), dtype=torch.bfloat16, device="cuda")
        wsb = moe.moe_ffn_workspace_size(rows, cfg.I, moe.MOE_BF16)
        ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
        moe.moe_expert_ffn(x_rows, None, i32(offs), n_phys, i32(p2l), rows, pw.struct(), None, 0, y, ws, wsb, err)
        return y

    os.environ["MOE_B300_FFN_TILES"] = mode
    try:
        whole = ffn(xp, po, P, p2l_all, N)
        per = P // cfg.R
        slices = []
        for r in range(cfg.R):
            a, b = int(po[r * per]), int(po[(r + 1) * per])
            assert a == lay["rank_offsets"][r] and b == lay["rank_offsets"][r + 1]
            if b > a:
                slices.append((a, b, ffn(xp[a:b], po[r * per:(r + 1) * per + 1] - a, per,
                                         p2l_all[r * per:(r + 1) * per], b - a)))
        torch.cuda.synchronize()
    finally:
        del os.environ["MOE_B300_FFN_TILES"]
    assert int(err.item()) == 0
    assert len(slices) > 1
    for a, b, y in slices:
        assert torch.equal(y[:b - a].view(torch.int16), whole[a:b].view(torch.int16))
