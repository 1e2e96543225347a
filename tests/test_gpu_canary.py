"""Out-of-bounds writes and run-to-run determinism, on the GPU.

Every device buffer a call writes -- the layer's workspace, its output and every
intermediate it exposes, and the outputs of the fused FFN entry points -- sits between
two 4 KB guard regions filled with 0xA5 bytes; after the call both guards must be
intact (a write past either end of any output would change them).  The layer runs
in every precision and tile orientation, with ragged tails.  The same inputs run
twice must give bit-identical outputs (no step of the layer depends on the order in
which threads finish)."""
import math

import numpy as np
import pytest
import torch

import combine_softmax_top_expert_b300 as moe
import moe_inputs as mi
from combine_softmax_top_expert_b300.layer import Layer, LayerAux, PackedWeights, dtype_code
from oracle import moe_oracle as O

from _util import dev_bf16, dev_f32, dev_x, fill_weights

pytestmark = pytest.mark.gpu
GUARD = 4096
FILL = 0xA5


class Guarded:
    """Device buffers with a guard region on each side."""

    def __init__(self):
        self.raw = []

    def alloc(self, shape, dtype):
        shape = tuple(shape) if isinstance(shape, (tuple, list)) else (shape,)
        n = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        raw = torch.full((n + 2 * GUARD,), FILL, dtype=torch.uint8, device="cuda")
        self.raw.append((raw, n))
        return raw[GUARD:GUARD + n].view(dtype).view(shape)

    def check(self):
        torch.cuda.synchronize()
        for i, (raw, n) in enumerate(self.raw):
            head, tail = raw[:GUARD], raw[GUARD + n:]
            assert bool((head == FILL).all()), f"buffer {i}: a write before its start"
            assert bool((tail == FILL).all()), f"buffer {i}: a write past its end ({n} bytes)"


def guarded_layer(cfg):
    """A Layer whose workspace, output and every exposed intermediate are guarded."""
    act = moe.MOE_F32 if cfg.dtype == "fp32" else moe.MOE_BF16
    ex = dtype_code(cfg.dtype)
    pw = PackedWeights(cfg.E, cfg.d, cfg.I, ex, cfg.shared)
    fill_weights(cfg, pw)
    layer = Layer(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.R, act, ex, cfg.shared, cfg.n_redundant, pw,
                  eplb_placement=cfg.eplb_placement, expert_placement=cfg.expert_placement,
                  fp8_dispatch=cfg.fp8_dispatch)
    g = Guarded()
    layer.ws = g.alloc(layer.ws_bytes, torch.uint8)
    layer.out = g.alloc(tuple(layer.out.shape), layer.out.dtype)
    for name, t in list(layer.bufs.items()):
        layer.bufs[name] = g.alloc(tuple(t.shape), t.dtype)
    layer.aux = LayerAux(**{n: t.data_ptr() for n, t in layer.bufs.items()})
    return layer, g


CASES = [
    ("fp32, ragged", mi.config("tiny_fp32").scaled(T=37)),
    ("bf16 + shared, pair gate/up and wide down (d = 384)",
     mi.config("prefill_bf16_skew").scaled(T=300, d=384, E=16, k=4, I=256, R=4)),
    ("bf16 decode-shaped: swap tiles", mi.config("decode_bf16").scaled(T=16, d=256, E=64, k=8, I=256, R=8)),
    ("bf16 + shared, load-aware EPLB, FP8 dispatch",
     mi.config("prefill_bf16_skew_eplb").scaled(T=512, d=512, E=32, k=8, I=256, R=8, n_redundant=8, eplb_placement=1,
                                                fp8_dispatch=1)),
    ("bf16, EPLB hottest replicas, round-robin placement",
     mi.config("prefill_bf16_skew_eplb").scaled(T=260, d=256, E=16, k=4, I=256, R=4, n_redundant=4,
                                                expert_placement=1)),
    ("e4m3 experts, pair tiles", mi.config("prefill_fp8_skew").scaled(T=400, d=512, E=16, k=4, I=256, R=4)),
    ("e4m3 experts, one-SM tiles", mi.config("prefill_fp8_skew").scaled(T=40, d=512, E=64, k=4, I=256, R=8)),
]


@pytest.mark.parametrize("name,cfg", CASES, ids=[c[0] for c in CASES])
def test_layer_writes_stay_inside_buffers_and_repeat_exactly(name, cfg):
    layer, g = guarded_layer(cfg)
    logits, x = dev_f32(mi.make_logits(cfg)), dev_x(cfg, mi.make_x(cfg))
    first = layer.forward(logits, x).clone()
    g.check()
    aux_first = {n: t.clone() for n, t in layer.bufs.items()}
    second = layer.forward(logits, x)
    g.check()
    assert int(layer.err.item()) == 0
    assert torch.equal(first.view(torch.uint8), second.view(torch.uint8))
    for n, t in layer.bufs.items():
        assert torch.equal(aux_first[n].view(torch.uint8), t.view(torch.uint8)), n


def test_fused_entry_points_write_inside_their_buffers():
    cfg = mi.config("prefill_bf16_skew").scaled(T=300, d=384, E=16, k=4, I=256, R=4)
    ids, tw = O.route(mi.make_logits(cfg), cfg.k)
    lay = O.dispatch_layout(ids, cfg.E, cfg.R, None)
    N, T = cfg.N, cfg.T
    pw = PackedWeights(cfg.E, cfg.d, cfg.I, moe.MOE_BF16, True)
    fill_weights(cfg, pw)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    offs, r2t, s2r = i32(lay["phys_offsets"]), i32(lay["row_to_token"]), i32(lay["slot_to_row"])
    twd = torch.from_numpy(np.ascontiguousarray(tw, dtype=np.float32)).cuda()
    x = dev_bf16(mi.make_x(cfg))
    g = Guarded()
    h = g.alloc((N + T, cfg.I), torch.bfloat16)
    y = g.alloc((N + T, cfg.d), torch.bfloat16)
    out = g.alloc((T, cfg.d), torch.bfloat16)
    counts = g.alloc(T * (cfg.d // 128), torch.int32)
    err = g.alloc(1, torch.int32)
    err.zero_()
    moe.moe_expert_gate_up_gather(x, T, r2t, offs, cfg.E, None, N, pw.struct(), x, T, h, err)
    moe.moe_expert_down_combine(h, offs, cfg.E, None, N, pw.struct(), T, r2t, s2r, twd, T, cfg.k, y, counts, out,
                                err)
    g.check()
    assert int(err.item()) == 0
