"""What the fp8 tolerances can see (no GPU): on the oracle's e4m3 expert FFN, a block
scale 5-10 % off on one of the 48 K blocks of d = 6144 moves the output by more than
the consistency bound the fp8 tests apply (1e-2 of rms(out)) and by less than the
method's 5e-2, so that check is the one that would catch it."""
import numpy as np
import pytest

import moe_inputs as mi
from oracle import moe_oracle as O

from _util import FP8_CONSISTENCY, FP8_RMS


@pytest.mark.parametrize("factor", [1.05, 1.1])
@pytest.mark.parametrize("block", [0, 30, 47])
def test_one_block_scale_slip_is_between_the_bounds(factor, block):
    cfg = mi.config("prefill_fp8_skew").scaled(T=64, E=1, k=1, I=256, R=1)
    x = mi.f32_from_bf16_bits(mi.make_x(cfg)).astype(np.float64)
    xq, xs = O.quantize_groups(x)
    w = {}
    for which in ("w_gate", "w_up", "w_down"):
        q, s = O.quantize_blocks(mi.f32_from_bf16_bits(mi.make_weight_host(cfg, which, 0)))
        w[which] = O.dequantize_blocks(q, s)

    def out(scales):
        return O.swiglu_expert(O.dequantize_groups(xq, scales), w["w_gate"], w["w_up"], w["w_down"], "fp8")

    ref = out(xs)
    slipped = xs.copy()
    slipped[:, block] *= factor
    shift = np.sqrt(np.mean((out(slipped) - ref) ** 2)) / np.sqrt(np.mean(ref ** 2))
    assert cfg.d // 128 == 48
    assert FP8_CONSISTENCY < shift < FP8_RMS, shift
