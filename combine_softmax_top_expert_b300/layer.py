"""Device-memory plumbing around the C ABI: packed weight sets, workspaces and
the intermediate buffers of moe_layer_forward, all allocated with torch.  No
arithmetic of the layer happens here."""
from __future__ import annotations

import torch

from . import (MOE_BF16, MOE_E4M3, MOE_F32, LayerAux, LoadStats, Shape, Weights, moe_layer_forward,
               moe_layer_workspace_size, moe_pack_weights)

_TORCH = {MOE_F32: torch.float32, MOE_BF16: torch.bfloat16, MOE_E4M3: torch.uint8}


def dtype_code(name: str) -> int:
    return {"fp32": MOE_F32, "f32": MOE_F32, "bf16": MOE_BF16, "fp8": MOE_E4M3, "e4m3": MOE_E4M3}[name]


class PackedWeights:
    """Packed expert weights (moe_weights_t) for E routed experts (+1 shared)."""

    def __init__(self, E, d, I, dtype: int, shared: bool, device="cuda", selection_bias=None):
        self.E, self.d, self.I, self.dtype, self.shared = E, d, I, dtype, shared
        self.selection_bias = selection_bias   # fp32 [E] on the device, or None
        self.E_w = E + (1 if shared else 0)
        t = _TORCH[dtype]
        self.w13 = torch.empty((self.E_w, 2 * I, d), dtype=t, device=device)
        self.w2 = torch.empty((self.E_w, d, I), dtype=t, device=device)
        self.s13 = self.s2 = None
        if dtype == MOE_E4M3:
            self.s13 = torch.empty((self.E_w, 2 * I // 128, d // 128), dtype=torch.float32, device=device)
            self.s2 = torch.empty((self.E_w, d // 128, I // 128), dtype=torch.float32, device=device)

    def pack(self, e, w_gate, w_up, w_down, stream=None):
        """Pack logical expert e (w_gate, w_up [d, I]; w_down [I, d]; fp32 or bf16)."""
        src = MOE_F32 if w_gate.dtype == torch.float32 else MOE_BF16
        moe_pack_weights(w_gate, w_up, w_down, src, self.d, self.I, self.dtype, self.w13[e], self.w2[e],
                         None if self.s13 is None else self.s13[e], None if self.s2 is None else self.s2[e],
                         stream)

    def struct(self) -> Weights:
        w = Weights()
        w.dtype, w.has_shared, w.E_w, w.d, w.I = self.dtype, int(self.shared), self.E_w, self.d, self.I
        w.w13, w.w2 = self.w13.data_ptr(), self.w2.data_ptr()
        w.s13 = self.s13.data_ptr() if self.s13 is not None else None
        w.s2 = self.s2.data_ptr() if self.s2 is not None else None
        w.selection_bias = self.selection_bias.data_ptr() if self.selection_bias is not None else None
        return w


class Layer:
    """moe_layer_forward with its workspace and (optionally) every intermediate
    exposed through moe_layer_aux_t."""

    def __init__(self, T, d, E, k, I, R, act_dtype, expert_dtype, shared=False, n_redundant=0,
                 weights: PackedWeights | None = None, keep_aux=True, device="cuda", eplb_placement=0,
                 expert_placement=0, fp8_dispatch=0):
        s = Shape()
        s.T, s.d, s.E, s.I, s.k, s.R = T, d, E, I, k, R
        s.n_redundant, s.shared, s.act_dtype, s.expert_dtype = n_redundant, int(shared), act_dtype, expert_dtype
        s.eplb_placement, s.expert_placement, s.fp8_dispatch = eplb_placement, expert_placement, fp8_dispatch
        self.shape, self.device = s, device
        self.weights = weights
        self.ws_bytes = moe_layer_workspace_size(s)
        if self.ws_bytes == 0:
            raise ValueError("shape rejected by moe_layer_workspace_size")
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.out = torch.empty((T, d), dtype=_TORCH[act_dtype], device=device)
        P, N = E + n_redundant, T * k
        self.aux = None
        self.bufs = {}
        if keep_aux:
            i32 = dict(dtype=torch.int32, device=device)
            b = self.bufs
            b["topk_ids"] = torch.empty((T, k), **i32)
            b["topk_w"] = torch.empty((T, k), dtype=torch.float32, device=device)
            b["logical_counts"] = torch.empty(E, **i32)
            b["phys_counts"] = torch.empty(P, **i32)
            b["phys_offsets"] = torch.empty(P + 1, **i32)
            b["rank_counts"] = torch.empty(R, **i32)
            b["rank_offsets"] = torch.empty(R + 1, **i32)
            b["row_to_token"] = torch.empty(N, **i32)
            b["slot_to_row"] = torch.empty((T, k), **i32)
            b["stats"] = torch.empty(2 * 8, **i32)
            b["phys_to_logical"] = torch.empty(P, **i32)
            b["phys_rank"] = torch.empty(P, **i32)
            b["replica_count"] = torch.empty(E, **i32)
            b["logical_to_phys"] = torch.empty((E, 1 + n_redundant if eplb_placement == 1 else 2), **i32)
            self.aux = LayerAux(**{n: t.data_ptr() for n, t in b.items()})

    def forward(self, logits, x, out=None, stream=None):
        out = self.out if out is None else out
        moe_layer_forward(self.shape, logits, x, self.weights.struct(), out, self.aux, self.ws, self.ws_bytes,
                          self.err, stream)
        return out

    def stats(self):
        """The two moe_load_stats_t records (before, after EPLB) as dicts."""
        raw = self.bufs["stats"].cpu().numpy().tobytes()
        out = []
        for i in range(2):
            st = LoadStats.from_buffer_copy(raw[32 * i:32 * (i + 1)])
            out.append({f: getattr(st, f) for f, _ in LoadStats._fields_ if not f.startswith("pad")})
        return out
