"""Block-scaled e4m3 expert FFN (moe_expert_ffn, weights e4m3 per 128x128 block,
activations e4m3 per row per 128 channels) and the fp8 layer against the oracle.
The tolerance is rms(gpu - oracle) <= 5e-2 * rms(oracle), checked over all outputs
and also row by row so that one wrong scale block cannot hide in the average."""
import os

import numpy as np
import pytest
import torch

import combine_softmax_top_expert_b300 as moe
import moe_inputs as mi
from combine_softmax_top_expert_b300.layer import PackedWeights
from oracle import moe_oracle as O

from _util import FP8_CONSISTENCY, FP8_RMS, fill_weights

pytestmark = pytest.mark.gpu


def rms(a):
    return float(np.sqrt(np.mean(np.square(a))))


def check_rms(got, ref, per_row=True):
    assert np.all(np.isfinite(got))
    err = rms(got - ref)
    print(f"rms error / rms(out) = {err / rms(ref):.3e}")
    assert err <= FP8_RMS * rms(ref), (err, rms(ref))
    assert err <= FP8_CONSISTENCY * rms(ref), (err, rms(ref))
    if per_row:
        row_err = np.sqrt(np.mean((got - ref) ** 2, axis=1))
        row_ref = np.sqrt(np.mean(ref ** 2, axis=1))
        bad = row_err > FP8_RMS * np.maximum(row_ref, 1e-6)
        assert not bad.any(), (int(bad.sum()), float(row_err.max()))
    return err / rms(ref)


def run_ffn_fp8(cfg, logits=None, mode=None):
    logits = mi.make_logits(cfg) if logits is None else logits
    ids, _ = O.route(logits, cfg.k)
    lay = O.dispatch_layout(ids, cfg.E, cfg.R)
    x = mi.f32_from_bf16_bits(mi.make_x(cfg))
    xq, xs = O.quantize_groups(x)                       # the permute's rule, per token
    r2t = lay["row_to_token"]
    pw = PackedWeights(cfg.E, cfg.d, cfg.I, moe.MOE_E4M3, False)
    fill_weights(cfg, pw)
    N = cfg.N
    y = torch.full((N, cfg.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    wsb = moe.moe_ffn_workspace_size(N, cfg.I, moe.MOE_E4M3)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    offs = torch.from_numpy(lay["phys_offsets"].astype(np.int32)).cuda()
    xq_d = torch.from_numpy(np.ascontiguousarray(xq[r2t])).cuda()
    xs_d = torch.from_numpy(np.ascontiguousarray(xs[r2t])).cuda()
    if mode:
        os.environ["MOE_B300_FFN_TILES"] = mode
    try:
        moe.moe_expert_ffn(xq_d, xs_d, offs, cfg.E, None, N, pw.struct(), None, 0, y, ws, wsb, err)
        torch.cuda.synchronize()
    finally:
        os.environ.pop("MOE_B300_FFN_TILES", None)
    assert int(err.item()) == 0
    got = y.float().cpu().numpy()
    xdeq = O.dequantize_groups(xq, xs)[r2t]
    ref = np.zeros((N, cfg.d))

    def W(which, e):
        q, s = O.quantize_blocks(mi.f32_from_bf16_bits(mi.make_weight_host(cfg, which, e)))
        return O.dequantize_blocks(q, s)

    for e in range(cfg.E):
        a, b = lay["phys_offsets"][e], lay["phys_offsets"][e + 1]
        if b > a:
            ref[a:b] = O.swiglu_expert(xdeq[a:b], W("w_gate", e), W("w_up", e), W("w_down", e), "fp8")
    return check_rms(got, ref)


SMALL = mi.config("prefill_fp8_skew").scaled(T=300, d=256, E=8, I=256, R=4)
MODES = ["wide", "pair"]      # one-SM tiles, SM-pair tiles


@pytest.mark.parametrize("mode", MODES)
def test_ffn_fp8_small(mode):
    run_ffn_fp8(SMALL, mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_ffn_fp8_skewed_groups_and_ragged_tiles(mode):
    cfg = SMALL.scaled(T=333, E=16, k=4, d=512, I=384, R=4)
    rng = np.random.default_rng(0)
    l = rng.standard_normal((cfg.T, cfg.E)).astype(np.float32)
    l[:, 2] += 6.0          # one expert takes nearly every token: many tiles, ragged tail
    l[:, 7] -= 20.0         # an expert that no token picks
    run_ffn_fp8(cfg, logits=l, mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_ffn_fp8_single_token(mode):
    run_ffn_fp8(SMALL.scaled(T=1), mode=mode)



@pytest.mark.parametrize("mode", MODES)
def test_ffn_fp8_one_k_block(mode):
    # I = 128: the down projection's only K block is also its first one
    run_ffn_fp8(SMALL.scaled(I=128), mode=mode)


def test_ffn_fp8_more_tiles_than_sm_pairs():
    # at least 128 down tiles of 256 x 256 for the GPU's SM pairs: each pair runs
    # several tiles, so part of a tile's outputs leaves after the next tile's first block
    cfg = SMALL.scaled(T=2048, d=1024, E=8, k=4, I=256)
    run_ffn_fp8(cfg, mode="pair")
